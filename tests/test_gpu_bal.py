"""Balanced extend: a one-wave batch of skewed lengths (the longest request at least twice the mean)
runs as segments planned on the device, on one CTA per SM; the CTA of a later segment first forms
the state at its start from the request's earlier keys and values.

Checked through the C ABI:
  * which batches take it: skewed ones (by the caller's max_seqlen) with a workspace, not even ones;
  * the plan the device leaves in the workspace: every request is covered once by contiguous
    segments that start on chunk boundaries, the last one flagged, the uneven batches really cut,
    at most two items per CTA, and the non-last segments dealt first;
  * outputs and final states against the fp64 oracle, element by element: the skewed bench
    workload, the varlen workload (8 requests of 512-4096 tokens, 16 heads, under a loose
    max_seqlen), a batch with empty, one-token and chunk-edge
    requests, and a nearly flat decay that carries thousands of tokens through the prologues;
  * tracking snapshots inside the first segment, exactly at a segment start, inside the last
    segment and at the request's end, written into a head-major output;
  * faulty requests in a balanced batch are reported and skipped, the others are computed;
  * the balanced and the plain schedule agree within the tolerance, repeated calls bit for bit,
    and slots that no request names keep their bytes.
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
C = 128
REC_INTS = 12       # one segment record: b, y0, len, slot, sp, tslot, nchunks, flags, a, nseg, 0, 0
F_VALID, F_PREFIX, F_LAST = 1, 2, 4


@pytest.fixture(autouse=True)
def _balanced_on():
    la.set_balanced(True)
    yield
    la.set_balanced(True)


def _lens(w):
    return (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).tolist()


def _run(w, balanced=True, out=None, track=None, state_idx=None, max_seqlen=None, pool0=None):
    """One extend call with its own workspace; returns (out, pool, workspace)."""
    la.set_balanced(balanced)
    lens = _lens(w)
    ms = max(lens) if max_seqlen is None else max_seqlen
    nbytes = la.extend_workspace_size(w.B, w.T, w.H, w.D, ms)
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    pool = (w.materialize_pool() if pool0 is None else pool0).to(DEV)
    if out is None:
        out = torch.full((w.T, w.H * w.D), 5.0, dtype=torch.bfloat16, device=DEV)
    kw = {}
    if track is not None:
        kw = dict(track_lens=torch.tensor(track[0], dtype=torch.int32, device=DEV),
                  track_state_idx=torch.tensor(track[1], dtype=torch.int32, device=DEV))
    idx = w.state_idx if state_idx is None else state_idx
    la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(w.H, w.layer_id, w.L).to(DEV),
              pool, idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV), out=out,
              max_seqlen=ms, workspace=ws, **kw)
    la.set_balanced(True)
    return out, pool, ws


def _plan(ws):
    """The device's plan from the start of the workspace: records in deal order."""
    head = ws[:16].cpu().view(torch.int32).tolist()
    nrec = head[0]
    recs = ws[16:16 + 4 * REC_INTS * nrec].cpu().view(torch.int32).view(nrec, REC_INTS).numpy()
    return recs


def _check_plan(w, recs, sms, faulty=()):
    lens = _lens(w)
    cu = w.cu_seqlens.tolist()
    assert len(recs) * w.H <= 2 * sms, "more than two items per CTA"
    nonlast = [i for i, r in enumerate(recs) if not r[7] & F_LAST]
    assert nonlast == list(range(len(nonlast))), "non-last segments must be dealt first"
    assert len(nonlast) * w.H <= sms, "a non-last segment is not the first item of its CTA"
    covered = set()
    for b in range(w.B):
        segs = sorted((r for r in recs if r[0] == b), key=lambda r: r[8])
        if b in faulty:
            assert not segs, f"faulty request {b} has a segment"
            continue
        covered.add(b)
        assert segs, f"request {b} has no segment"
        a = 0
        for j, r in enumerate(segs):
            _, y0, ln, slot, sp, tslot, nch, flags, ra, nseg = r[:10]
            assert ra == a and ra % C == 0, f"request {b}: segment {j} starts at {ra}, not {a}"
            assert y0 == cu[b] + ra and slot == int(w.state_idx[b]) and nseg == len(segs)
            assert flags & F_VALID and bool(flags & F_PREFIX) == bool(w.prefix_mask[b])
            assert bool(flags & F_LAST) == (j + 1 == len(segs))
            assert ln >= 0 and (ln > 0 or len(segs) == 1)
            a += ln
        assert a == lens[b], f"request {b}: segments cover {a} of {lens[b]} tokens"
    return sum(1 for b in covered if sum(1 for r in recs if r[0] == b) > 1)


def _oracle(w, pool0, track=None):
    args = (w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
            oracle_slopes_fp32(w.H, w.layer_id, w.L), pool0.double().numpy(), w.state_idx.numpy(),
            w.cu_seqlens.numpy(), w.prefix_mask.numpy())
    if track is None:
        return oracle.extend(*args, w.H, w.D)
    return oracle.extend_tracked(*args, np.asarray(track[0], dtype=np.int32),
                                 np.asarray(track[1], dtype=np.int32), w.H, w.D)


def _sms():
    return torch.cuda.get_device_properties(DEV).multi_processor_count


def _check_states(w, pool, pool0, p_ref, extra=(), what=""):
    pa = pool.cpu()
    named = sorted(set(w.state_idx.tolist()) | set(extra))
    assert_close(pa.double().numpy()[named], p_ref[named], f"{what}: states")
    untouched = np.ones(w.num_slots, bool)
    untouched[named] = False
    u = torch.from_numpy(untouched)
    assert torch.equal(pa[u].view(torch.int32), pool0[u].view(torch.int32)), \
        f"{what}: an unnamed slot changed"


def test_only_skewed_one_wave_batches_take_it():
    w = workloads.varlen_extend()
    lens = _lens(w)
    # lengths within a factor of two of the mean: the column split serves them, no plan needed
    assert la.extend_workspace_size(w.B, w.T, w.H, w.D, max(lens)) == 0
    # the same batch under a looser bound counts as skewed and gets a plan
    assert la.extend_workspace_size(w.B, w.T, w.H, w.D, w.T) > 0
    # more (request, head) pairs than SMs: the persistent grid's records only (32 bytes a request)
    sms = _sms()
    assert la.extend_workspace_size(sms, sms * 64, 2, 128, sms * 64) == 32 * sms


def test_varlen_workload_balanced_against_the_oracle():
    """The varlen workload with max_seqlen = T: counted as skewed, so it runs balanced."""
    w = workloads.varlen_extend()
    assert w.B * w.H <= _sms()
    pool0 = w.materialize_pool()
    out, pool, ws = _run(w, max_seqlen=w.T)
    la.poll_error()
    assert _check_plan(w, _plan(ws), _sms()) >= 1, "the longest request was not cut"
    o_ref, p_ref = _oracle(w, pool0)
    assert_close(to64(out), o_ref, "varlen balanced: out")
    _check_states(w, pool, pool0, p_ref, what="varlen balanced")
    # the same call again gives the same bits; the plain schedule agrees within the tolerance
    out2, pool2, _ = _run(w, max_seqlen=w.T)
    assert torch.equal(out2, out) and torch.equal(pool2.view(torch.int32), pool.view(torch.int32))
    out0, pool0_run, ws0 = _run(w, balanced=False, max_seqlen=w.T)
    la.poll_error()
    assert_close(to64(out0), to64(out), "balanced against plain: out")


@pytest.mark.parametrize("layer_id,L", [(0, 1), (7, 8)], ids=["steep", "nearly_flat"])
def test_ragged_batch_with_edge_lengths(layer_id, L):
    """Empty, one-token and chunk-edge requests next to long ones; with layer 7 of 8 the slopes
    are about 1e-5 of the ALiBi base, so the prologue carries thousands of tokens of memory."""
    lens = [3000, 40, 0, 1, 2500, 129, 128, 1800, 700, 2047, 0, 3333]
    prefix = [1, 0, 1, 0, 1, 1, 0, 0, 1, 0, 0, 1]
    w = workloads.custom_extend(lens, H=8, prefix=prefix, layer_id=layer_id, L=L, seed=41,
                                num_slots=40)
    pool0 = w.materialize_pool()
    out, pool, ws = _run(w)
    la.poll_error()
    assert _check_plan(w, _plan(ws), _sms()) >= 1
    o_ref, p_ref = _oracle(w, pool0)
    assert_close(to64(out), o_ref, "ragged balanced: out")
    _check_states(w, pool, pool0, p_ref, what="ragged balanced")


def test_snapshots_at_segment_boundaries_and_head_major_output():
    lens = [6000, 600, 2900, 1500, 3100, 256, 900, 2200]
    w = workloads.custom_extend(lens, H=16, prefix=[b % 2 == 0 for b in range(8)], layer_id=1,
                                L=4, seed=43, num_slots=48)
    assert max(lens) * w.B >= 2 * w.T, "the batch must count as skewed"
    _, _, ws = _run(w)
    la.poll_error()
    recs = _plan(ws)
    assert _check_plan(w, recs, _sms()) >= 1
    # track lengths: a segment start of every cut request, else inside, at the end, 0, none
    tl = []
    for b, n in enumerate(lens):
        starts = sorted(int(r[8]) for r in recs if r[0] == b and r[8] > 0)
        if starts and b % 2 == 0:
            tl.append(starts[0])
        elif starts:
            tl.append(starts[-1] + 77)
        else:
            tl.append([n, 0, -1, n // 3][b % 4])
    used = set(w.state_idx.tolist())
    free = [s for s in range(w.num_slots) if s not in used]
    ti = [free[b] for b in range(w.B)]
    pool0 = w.materialize_pool()
    hm = torch.full((w.H, w.T, w.D), 3.0, dtype=torch.bfloat16, device=DEV)
    _, pool, ws2 = _run(w, out=hm.transpose(0, 1), track=(tl, ti), pool0=pool0)
    la.poll_error()
    assert np.array_equal(_plan(ws2)[:, [0, 1, 2, 8]], recs[:, [0, 1, 2, 8]]), \
        "the plan must not depend on tracking"
    o_ref, p_ref = _oracle(w, pool0, track=(tl, ti))
    got = to64(hm.transpose(0, 1).reshape(w.T, w.H * w.D))
    assert_close(got, o_ref, "balanced tracked: out")
    _check_states(w, pool, pool0, p_ref, extra=[t for t, x in zip(ti, tl) if x >= 0],
                  what="balanced tracked")


def test_faulty_requests_in_a_balanced_batch():
    """A slot out of range and a request over max_seqlen: reported, nothing of them written; the
    plan leaves them out and the other requests match the oracle."""
    lens = [2600, 300, 400, 4000, 700, 200]
    w = workloads.custom_extend(lens, H=16, prefix=[1, 0, 1, 1, 0, 1], seed=47, num_slots=24)
    idx = w.state_idx.clone()
    idx[1] = w.num_slots + 2
    cap = 3000  # request 3 (4000 tokens) exceeds it; the batch still counts as skewed
    assert cap * w.B >= 2 * w.T
    pool0 = w.materialize_pool()
    out, pool, ws = _run(w, state_idx=idx, max_seqlen=cap, pool0=pool0)
    with pytest.raises(la.LAError) as e:
        la.poll_error()
    assert e.value.status == 5
    la.poll_error()
    recs = _plan(ws)
    assert _check_plan(w, recs, _sms(), faulty=(1, 3)) >= 1
    cu = w.cu_seqlens.tolist()
    for b in (1, 3):
        assert (out[cu[b]:cu[b + 1]] == 5.0).all(), f"request {b} wrote output rows"
    assert torch.equal(pool.cpu()[int(w.state_idx[3])].view(torch.int32),
                       pool0[int(w.state_idx[3])].view(torch.int32))
    o_ref, p_ref = _oracle(w, pool0)
    ok = [b for b in range(w.B) if b not in (1, 3)]
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in ok])
    assert_close(to64(out)[rows], o_ref[rows], "balanced with faults: out")
    slots = [int(w.state_idx[b]) for b in ok]
    assert_close(pool.cpu().double().numpy()[slots], p_ref[slots], "balanced with faults: states")


def test_skewed_workload_against_the_oracle():
    """The bench's skewed workload (two requests of 4096-8192 tokens among six of 256-1024, 16
    heads) at full size: it takes the balanced schedule by its own max_seqlen, cuts the long
    requests, and matches the oracle element by element."""
    w = workloads.varlen_extend_skewed()
    lens = _lens(w)
    assert max(lens) * w.B >= 2 * w.T and w.B * w.H <= _sms()
    pool0 = w.materialize_pool()
    out, pool, ws = _run(w)
    la.poll_error()
    recs = _plan(ws)
    assert _check_plan(w, recs, _sms()) >= 2, "both long requests should be cut"
    o_ref, p_ref = _oracle(w, pool0)
    assert_close(to64(out), o_ref, "skewed workload: out")
    _check_states(w, pool, pool0, p_ref, what="skewed workload")


def _draw_skewed(seed):
    """A random skewed one-wave batch: 5-9 requests, 12 or 16 heads (so that B H fills more than
    half of 152 SMs and no sequence split is planned), one or two of 1500-5000 tokens, the rest 0-700
    with chunk edges; caller slopes log-uniform over six decades (some exactly zero)."""
    rng = np.random.default_rng(5000 + seed)
    B = int(rng.integers(5, 10))
    H = int(rng.choice([12, 16])) if B >= 7 else 16  # B H > 76: more than half the SMs
    edges = [0, 1, 127, 128, 129, 255, 256, 511]
    lengths = [int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(0, 700))
               for _ in range(B)]
    for i in rng.choice(B, size=int(rng.integers(1, 3)), replace=False):
        lengths[int(i)] = int(rng.integers(1500, 5001))
    top = int(np.argmax(lengths))
    while lengths[top] * B < 2 * sum(lengths):  # skewed: the longest at least twice the mean
        lengths[top] += 512
    slopes = np.where(rng.random(H) < 0.15, 0.0, 10.0 ** rng.uniform(-6, np.log10(3), H))
    prefix = [int(x) for x in rng.integers(0, 2, B)]
    return rng, lengths, H, slopes.astype(np.float32), prefix


@pytest.mark.parametrize("seed", range(8))
def test_balanced_fuzz(seed):
    """Random skewed batches with tracking snapshots at random offsets and the three output
    layouts, against the oracle, with a valid plan."""
    rng, lengths, H, slopes, prefix = _draw_skewed(seed)
    B = len(lengths)
    w = workloads.custom_extend(lengths, H=H, prefix=prefix, num_slots=2 * B + 2, seed=seed)
    T = w.T
    assert max(lengths) * B >= 2 * T and B * H <= _sms()
    tl = np.array([int(rng.integers(0, n + 1)) if rng.random() < 0.7 else -1 for n in lengths],
                  dtype=np.int32)
    used = set(int(x) for x in w.state_idx.numpy())
    free = [s for s in range(w.num_slots) if s not in used]
    ti = np.array([free[b] if tl[b] >= 0 else -1 for b in range(B)], dtype=np.int32)
    layout = ["packed", "per_head", "head_major"][seed % 3]
    if layout == "head_major":
        buf = torch.full((H, T, 128), 3.0, dtype=torch.bfloat16, device=DEV)
        view = buf.transpose(0, 1)
    elif layout == "per_head":
        view = torch.full((T, H, 128), 3.0, dtype=torch.bfloat16, device=DEV)
    else:
        view = torch.full((T, H * 128), 3.0, dtype=torch.bfloat16, device=DEV)
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    nbytes = la.extend_workspace_size(B, T, H, 128, max(lengths))
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), torch.from_numpy(slopes).to(DEV), pool,
              w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV), out=view,
              max_seqlen=max(lengths), workspace=ws, track_lens=torch.from_numpy(tl).to(DEV),
              track_state_idx=torch.from_numpy(ti).to(DEV))
    la.poll_error()
    _check_plan(w, _plan(ws), _sms())
    o_ref, p_ref = oracle.extend_tracked(w.q.float().numpy(), w.k.float().numpy(),
                                         w.v.float().numpy(), slopes.astype(np.float64),
                                         pool0.double().numpy(), w.state_idx.numpy(),
                                         w.cu_seqlens.numpy(), w.prefix_mask.numpy(), tl, ti, H,
                                         128)
    tag = f"seed {seed} (B={B} H={H} lengths={lengths} {layout})"
    assert_close(to64(view.reshape(T, H * 128)), o_ref, f"{tag}: out")
    _check_states(w, pool, pool0, p_ref, extra=[int(x) for x in ti if x >= 0], what=tag)


def test_balanced_graph_replay():
    """The plan kernel and the balanced grid captured in a CUDA graph: two replays on new inputs
    equal the eager calls bit for bit."""
    lengths = [2600, 300, 400, 200, 700, 150]
    w = workloads.custom_extend(lengths, H=16, prefix=[1, 0, 1, 0, 1, 1], seed=29, num_slots=16)
    s = la.slopes(w.H, w.layer_id, w.L).to(DEV)
    T, ms = w.T, max(lengths)
    nbytes = la.extend_workspace_size(w.B, T, w.H, w.D, ms)
    assert 0 < nbytes < 65536, "the batch must take the balanced schedule"
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    pool0 = w.materialize_pool()
    qs, ks, vs = (torch.zeros(T, w.H * w.D, dtype=torch.bfloat16, device=DEV) for _ in range(3))
    out = torch.empty(T, w.H * w.D, dtype=torch.bfloat16, device=DEV)
    pool_g = pool0.to(DEV)
    idx_d, cu_d, pm_d = w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV)
    # warm-up outside the capture (module load, attributes)
    la.extend(qs, ks, vs, s, pool0.to(DEV), idx_d, cu_d, pm_d, max_seqlen=ms, workspace=ws)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            la.extend(qs, ks, vs, s, pool_g, idx_d, cu_d, pm_d, out=out, max_seqlen=ms,
                      workspace=ws)
    la.poll_error()
    for step in range(2):
        gen = torch.Generator().manual_seed(700 + step)
        q, k, v = (torch.randn(T, w.H * w.D, generator=gen).to(torch.bfloat16) for _ in range(3))
        pool_g.copy_(pool0.to(DEV))
        qs.copy_(q)
        ks.copy_(k)
        vs.copy_(v)
        g.replay()
        torch.cuda.synchronize()
        pool_e = pool0.to(DEV)
        o_e = la.extend(q.to(DEV), k.to(DEV), v.to(DEV), s, pool_e, idx_d, cu_d, pm_d,
                        max_seqlen=ms, workspace=ws)
        la.poll_error()
        assert torch.equal(out.cpu(), o_e.cpu()), f"step {step}: replay != eager output"
        assert torch.equal(pool_g.cpu().view(torch.int32), pool_e.cpu().view(torch.int32))


def test_many_requests_one_head():
    """150 one-head requests (one of 6000 tokens among short ones): the planner walks the
    requests 32 at a time in every warp, and records stay within the limits."""
    rng = np.random.default_rng(31)
    lens = [int(x) for x in rng.integers(0, 300, size=150)]
    lens[77] = 6000
    w = workloads.custom_extend(lens, H=1, prefix=[b % 3 == 0 for b in range(150)], seed=33,
                                num_slots=160)
    assert max(lens) * w.B >= 2 * w.T and w.B * w.H <= _sms()
    pool0 = w.materialize_pool()
    out, pool, ws = _run(w)
    la.poll_error()
    assert _check_plan(w, _plan(ws), _sms()) >= 1
    o_ref, p_ref = _oracle(w, pool0)
    assert_close(to64(out), o_ref, "150 requests, one head: out")
    _check_states(w, pool, pool0, p_ref, what="150 requests, one head")

"""GPU checks of the extend output layouts (la_extend_ex's output strides).

The page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析" (section
"生产环境不支持", item 4) describes the mismatch: the backend flattens out to [T, H*D] while the
piecewise-CUDA-graph path hands it a per-head [T, H, D] buffer.  Here out may be a per-head
buffer, a slice of a wider buffer or a head-major buffer seen through a transpose; every layout
must receive exactly the packed call's values (same kernel arithmetic, only the stores move) and
leave the bytes between the written elements untouched.
"""
import pytest
import torch

import lightning_attention_gb300 as la
from lightning_attention_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
CANARY = -77.0


def _inputs(w):
    return (w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(w.H, w.layer_id, w.L).to(DEV),
            w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV))


def _extend(w, out, **kw):
    q, k, v, s, idx, cu, pm = _inputs(w)
    pool = w.materialize_pool(DEV)
    ret = la.extend(q, k, v, s, pool, idx, cu, pm, out=out, **kw)
    la.poll_error()
    return ret, pool


def _layouts(T, H, D):
    """(name, full buffer, out view) triples; the view's elements are what the call writes."""
    per_head = torch.full((T, H, D), CANARY, dtype=torch.bfloat16, device=DEV)
    wide = torch.full((T, (H + 3) * D + 8), CANARY, dtype=torch.bfloat16, device=DEV)
    gapped = torch.full((T, H, D + 64), CANARY, dtype=torch.bfloat16, device=DEV)
    head_major = torch.full((H, T, D), CANARY, dtype=torch.bfloat16, device=DEV)
    return [("per_head", per_head, per_head),
            ("wide_rows", wide, wide[:, 2 * D + 8: 2 * D + 8 + H * D]),
            ("gapped_heads", gapped, gapped[:, :, :D]),
            ("head_major", head_major, head_major.transpose(0, 1))]


@pytest.mark.parametrize("lengths", [[300, 77, 1000, 0, 129], [5000, 3000]],
                         ids=["varlen", "split"])
def test_output_layouts_match_packed(lengths):
    w = workloads.custom_extend(lengths, H=3, layer_id=1, L=3, num_slots=16, seed=41)
    ref, pool_ref = _extend(w, None)
    ref3 = ref.view(w.T, w.H, w.D).cpu()
    for name, full, view in _layouts(w.T, w.H, w.D):
        before = full.clone()
        ret, pool = _extend(w, view)
        assert ret.data_ptr() == view.data_ptr()
        got = view.reshape(w.T, w.H, w.D).cpu() if view.dim() == 3 else view.cpu().view(
            w.T, w.H, w.D)
        assert torch.equal(got, ref3), f"{name}: values differ from the packed call"
        assert torch.equal(pool.cpu(), pool_ref.cpu()), f"{name}: states differ"
        # everything outside the view keeps its canary
        mask = torch.ones_like(full, dtype=torch.bool)
        if name == "wide_rows":
            mask[:, 2 * w.D + 8: 2 * w.D + 8 + w.H * w.D] = False
        elif name == "gapped_heads":
            mask[:, :, :w.D] = False
        else:
            mask[:] = False
        assert torch.equal(full[mask].cpu(), before[mask].cpu()), f"{name}: wrote outside out"


def test_layout_with_state_tracking():
    w = workloads.custom_extend([700, 260], H=2, num_slots=8, seed=42)
    used = set(w.state_idx.tolist())
    free = [s for s in range(w.num_slots) if s not in used][:2]
    tl = torch.tensor([333, 128], dtype=torch.int32, device=DEV)
    ti = torch.tensor(free, dtype=torch.int32, device=DEV)
    ref, pool_ref = _extend(w, None, track_lens=tl, track_state_idx=ti)
    _, full, view = _layouts(w.T, w.H, w.D)[3]
    _, pool = _extend(w, view, track_lens=tl, track_state_idx=ti)
    assert torch.equal(view.reshape(w.T, w.H, w.D).cpu(), ref.view(w.T, w.H, w.D).cpu())
    assert torch.equal(pool.cpu(), pool_ref.cpu())


def test_bad_layouts_rejected():
    w = workloads.custom_extend([64], H=2, num_slots=4, seed=43)
    odd = torch.empty((w.T, w.H * w.D + 4), dtype=torch.bfloat16, device=DEV)[:, 4:]
    with pytest.raises(la.LAError) as e:       # row stride H*D + 4: not a multiple of 8
        _extend(w, odd)
    assert e.value.status == 1
    with pytest.raises(ValueError):
        _extend(w, torch.empty((w.T, w.H * w.D), dtype=torch.bfloat16, device=DEV).t().t()[:, ::2])

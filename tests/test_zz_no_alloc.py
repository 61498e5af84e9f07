"""The allocation-free entry point, for callers that cannot allocate device memory where
they orthogonalize (a host framework's caching allocator owns the pool, a latency-critical
loop, a plugin that may not allocate): its results must match muon_orthogonalize_full,
which uses a caller-allocated workspace, on two calls in a row that share the static
scratch array.  This file is collected last on purpose."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from muon_optimizer_step_gb300 import inputs  # noqa: E402

TOL_NS_FP32 = 1e-4


@pytest.fixture(scope="module")
def capi():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from muon_optimizer_step_gb300 import capi as c
    return c


def _full_input(wl, layout, seed):
    g = inputs.host_grads(wl, seed)
    full = np.zeros(layout.full_numel, dtype=np.float32)
    pos = 0
    for i, (r, c) in enumerate(wl.shapes):
        if wl.is_matrix[i]:
            off = layout.full_offsets[i]
            full[off:off + r * c] = g[pos:pos + r * c] * (1.0 + i)
        pos += r * c
    return torch.from_numpy(full).cuda()


def _rel_per_matrix(a, b, wl, layout):
    a = a.cpu().numpy().astype(np.float64)
    b = b.cpu().numpy().astype(np.float64)
    out = []
    for i, (r, c) in enumerate(wl.shapes):
        if wl.is_matrix[i]:
            off = layout.full_offsets[i]
            x, y = a[off:off + r * c], b[off:off + r * c]
            out.append(float(np.linalg.norm(x - y) / np.linalg.norm(y)))
    return out


def test_noalloc_matches_allocating_entry_point_twice(capi):
    wl = inputs.WORKLOADS["ragged_small"]
    lay = capi.muon_layout_create(wl.shapes, 1, capi.MUON_NS_FP32, wl.is_matrix)
    ws = capi.workspace_tensor(lay)
    for call, seed in enumerate((0, 1)):
        fin = _full_input(wl, lay, seed)
        want = torch.zeros(lay.full_numel, device="cuda")
        capi.muon_orthogonalize_full(lay, ws, fin, want, 5)
        got = torch.full((lay.full_numel,), float("nan"), device="cuda")
        capi.muon_orthogonalize_full_noalloc(lay, fin, got, 5)
        capi.muon_check()
        errs = _rel_per_matrix(got, want, wl, lay)
        assert max(errs) < TOL_NS_FP32, (call, errs)


def test_noalloc_rejects_what_it_cannot_hold(capi):
    big = capi.muon_layout_create([(2048, 2048)], 1, capi.MUON_NS_FP32)
    fin = torch.zeros(big.full_numel, device="cuda")
    with pytest.raises(capi.MuonError) as e:
        capi.muon_orthogonalize_full_noalloc(big, fin, fin, 5)
    assert e.value.status == capi.MUON_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
    bf16 = capi.muon_layout_create([(8, 8)], 1, capi.MUON_NS_BF16)
    x = torch.zeros(64, device="cuda")
    with pytest.raises(capi.MuonError) as e:
        capi.muon_orthogonalize_full_noalloc(bf16, x, x, 5)
    assert e.value.status == capi.MUON_ERR_UNSUPPORTED

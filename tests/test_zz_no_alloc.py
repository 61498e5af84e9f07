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


def test_noalloc_zero_iterations_and_a_layout_near_the_limit(capi):
    """ns_steps = 0 (the export reads the input with the pending 1/||X|| scaling): equal
    to the allocating entry point and to the oracle's X / ||X||_F.  Then the largest
    square fp32 matrix whose tables and workspace still fit the scratch array, where the
    workspace ends closest to the array's end: equal to the allocating entry point."""
    from oracle import muon_ref as ref
    wl = inputs.WORKLOADS["ragged_small"]
    lay = capi.muon_layout_create(wl.shapes, 1, capi.MUON_NS_FP32, wl.is_matrix)
    ws = capi.workspace_tensor(lay)
    fin = _full_input(wl, lay, 3)
    want = torch.zeros(lay.full_numel, device="cuda")
    capi.muon_orthogonalize_full(lay, ws, fin, want, 0)
    got = torch.full((lay.full_numel,), float("nan"), device="cuda")
    capi.muon_orthogonalize_full_noalloc(lay, fin, got, 0)
    capi.muon_check()
    assert max(_rel_per_matrix(got, want, wl, lay)) < TOL_NS_FP32
    g = got.cpu().numpy().astype(np.float64)
    f = fin.cpu().numpy().astype(np.float64)
    for i, (r, c) in enumerate(wl.shapes):
        if wl.is_matrix[i]:
            off = lay.full_offsets[i]
            x = f[off:off + r * c].reshape(r, c)
            o = g[off:off + r * c].reshape(r, c)
            want_i = ref.newton_schulz(x, 0)  # X / ||X||_F, unit Frobenius norm
            assert np.linalg.norm(o - want_i) < 1e-5, (i, np.linalg.norm(o - want_i))
    # the largest n x n fp32 layout the array takes
    limit = 32 << 20
    for n in range(1448, 1300, -8):
        big = capi.muon_layout_create([(n, n)], 1, capi.MUON_NS_FP32)
        x = torch.randn(n * n, device="cuda") * 1e-3
        out = torch.full((n * n,), float("nan"), device="cuda")
        try:
            capi.muon_orthogonalize_full_noalloc(big, x, out, 5)
        except capi.MuonError as e:
            assert e.status == capi.MUON_ERR_UNSUPPORTED
            continue
        assert big.workspace_bytes > limit - (1 << 20), (n, big.workspace_bytes)
        ws_big = capi.workspace_tensor(big)
        ref_out = torch.zeros(n * n, device="cuda")
        capi.muon_orthogonalize_full(big, ws_big, x, ref_out, 5)
        capi.muon_check()
        e = float(torch.linalg.vector_norm((out - ref_out).double()) /
                  torch.linalg.vector_norm(ref_out.double()))
        assert e < TOL_NS_FP32, (n, e)
        break
    else:
        pytest.fail("no square layout fits the scratch array")

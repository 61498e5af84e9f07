"""GPU parity through muon_step on the GPT-2-small and mixture-of-experts matrix sets.

Newton-Schulz is per matrix on the owner ("Add initial Muon+M-FSDPv2 implementation",
"Opt step" step 4; FsdpMuon._orthogonalize_updates on the Megatron-Core API page), so
each set runs the whole optimizer step once, through the two calls muon_step makes
(momentum inputs, then orthogonalization with the apply fused into the last Update), and
the tests check:

* momentum and weights element by element (tests/parity.py bounds);
* the stored orthogonalization input element by element;
* the update O of the checked matrices against the oracle's Newton-Schulz of the GPU's
  own input: whole matrix, every 128 x 128 tile and every element;
* that muon_step itself gives the same bits as the two calls.

GPT-2-small (48 matrices: 768 x 2304, 768 x 768, 768 x 3072, 3072 x 768) exercises the
short reductions (K = 768) and m = 768 = 3 tiles.  The MoE set (64 experts of 2048 x 1408,
2048 x 1408 and 1408 x 2048, plus four dense 2048 x 2048) exercises 1408 = 5.5 x 256
columns, the half tile at the edge, and expert gradients scaled lognormally: the largest-
and smallest-scale experts' three matrices and one dense matrix are checked (Newton-Schulz
is scale invariant, so the scales must not move O).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle import muon_ref as ref  # noqa: E402
from muon_optimizer_step_gb300 import inputs  # noqa: E402
from tests import parity  # noqa: E402


@pytest.fixture(scope="module")
def capi():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from muon_optimizer_step_gb300 import capi as c
    return c


def _step_and_check(capi, wl, W0, G0, check_params, sample=None):
    """One step from M0 = 0; returns nothing, asserts everything.  W0, G0: flat fp32 CUDA
    tensors (left unchanged)."""
    lay = capi.muon_layout_create(wl.shapes, 1, capi.MUON_NS_BF16, wl.is_matrix)
    kern = capi.muon_layout_ns_kernel(lay)
    N = lay.numel
    ws = capi.workspace_tensor(lay)
    W = W0.clone()
    M = torch.zeros(N, device="cuda")
    fin = torch.zeros(lay.full_numel, device="cuda")
    fout = torch.zeros(lay.full_numel, device="cuda")
    capi.muon_compute_momentum_inputs([G0], [M], lay, ws, wl.mu, wl.nesterov)
    capi.muon_export_input(lay, ws, fin)
    capi.muon_orthogonalize_apply([W], lay, ws, wl.lr, wl.wd, wl.ns_steps)
    capi.muon_export_update(lay, ws, wl.ns_steps, fout)
    # muon_step on fresh copies: the same two calls, so the same bits
    W2 = W0.clone()
    M2 = torch.zeros(N, device="cuda")
    capi.muon_step([W2], [G0], [M2], lay, ws, wl.lr, wl.wd, wl.mu, wl.nesterov, wl.ns_steps)
    capi.muon_check()
    assert torch.equal(W2, W) and torch.equal(M2, M)
    del W2, M2

    offs = np.concatenate([[0], np.cumsum([r * c for r, c in wl.shapes])])
    if sample is None:
        sel = torch.arange(N, device="cuda")
    else:
        sel = torch.from_numpy(sample).cuda()
    g_s = G0[sel].double().cpu().numpy()
    w0_s = W0[sel].double().cpu().numpy()
    m_s = M[sel].double().cpu().numpy()
    w_s = W[sel].double().cpu().numpy()
    # momentum (M0 = 0): M1 = G
    parity.check_momentum(m_s, ref.momentum_update(np.zeros_like(g_s), g_s, wl.mu), 0.0,
                          wl.name)
    # weights against the oracle's decay and apply of the GPU's stored O (the fused tail
    # applies the fp32 O before its bf16 rounding: lr * s * 2^-8 * |O| more per element)
    flat = sel.cpu().numpy()
    owner = np.searchsorted(offs[1:], flat, side="right")
    full_pos = np.array(lay.full_offsets)[owner] + (flat - offs[owner])
    o_s = fout[torch.from_numpy(full_pos).cuda()].double().cpu().numpy()
    scale = np.array([ref.update_scale(*wl.shapes[j]) for j in range(len(wl.shapes))])[owner]
    lrs_o = wl.lr * scale * o_s
    want_w = ref.weight_decay(w0_s, wl.lr, wl.wd) - lrs_o
    parity.check_weights(w_s, want_w, w0_s, 1 - wl.lr * wl.wd, lrs_o,
                         extra=parity.BF16_REL * np.abs(lrs_o), what=(wl.name, kern))
    # inputs and Newton-Schulz of the checked matrices
    reports = []
    for i in check_params:
        r, c = wl.shapes[i]
        g = G0[offs[i]: offs[i + 1]].double().cpu().numpy()
        x_ref = ref.ns_input(g, ref.momentum_update(np.zeros_like(g), g, wl.mu), wl.mu,
                             wl.nesterov)
        off = lay.full_offsets[i]
        X = fin[off: off + r * c].double().cpu().numpy()
        parity.check_input(X, x_ref, g, 0, (wl.name, i))
        O = fout[off: off + r * c].view(r, c).double().cpu().numpy()
        rep = parity.check_ns(O, ref.newton_schulz(X.reshape(r, c), wl.ns_steps), 0,
                              (wl.name, i, (r, c), kern))
        reports.append((i, (r, c), rep))
    return reports


def test_gpt2_small_every_matrix(capi):
    wl = inputs.WORKLOADS["gpt2_small_x12"]
    W0, Gs, _ = inputs.host_inputs(wl)
    W0 = torch.from_numpy(W0).cuda()
    G0 = torch.from_numpy(Gs[0]).cuda()
    reps = _step_and_check(capi, wl, W0, G0, wl.matrix_indices())
    assert len(reps) == 48


def test_gpt2_input_rebuilt_on_the_host_bit_for_bit(capi):
    """With M0 = 0 the Nesterov input is fp32(0.95f * G + G) (one fused multiply-add)
    rounded to bf16: the host rebuild the full-size fused test relies on equals the stored
    input bit for bit."""
    wl = inputs.WORKLOADS["gpt2_small_x12"]
    _, Gs, _ = inputs.host_inputs(wl)
    lay = capi.muon_layout_create(wl.shapes, 1, capi.MUON_NS_BF16, wl.is_matrix)
    ws = capi.workspace_tensor(lay)
    G = torch.from_numpy(Gs[0]).cuda()
    M = torch.zeros_like(G)
    fin = torch.zeros(lay.full_numel, device="cuda")
    capi.muon_compute_momentum_inputs([G], [M], lay, ws, wl.mu, True)
    capi.muon_export_input(lay, ws, fin)
    capi.muon_check()
    mu32 = np.float64(np.float32(wl.mu))
    g = Gs[0].astype(np.float64)
    host = parity.bf16_round((mu32 * g + g).astype(np.float32))
    f = fin.cpu().numpy()
    pos = 0
    for i, (r, c) in enumerate(wl.shapes):
        off = lay.full_offsets[i]
        assert np.array_equal(f[off: off + r * c], host[pos: pos + r * c]), i
        pos += r * c


def test_moe_extreme_experts_and_dense(capi):
    wl = inputs.WORKLOADS["moe_64e"]
    N = wl.numel
    W0 = torch.zeros(N, device="cuda")
    G0 = torch.zeros(N, device="cuda")
    inputs.device_fill_weights(wl, W0)
    inputs.device_fill_grads(wl, G0, 0)
    offs = np.concatenate([[0], np.cumsum([r * c for r, c in wl.shapes])])
    # expert scale = norm of its gate gradient (all three share the lognormal factor)
    norms = [float(torch.linalg.vector_norm(G0[offs[3 * e]: offs[3 * e + 1]])) for e in range(64)]
    big, small = int(np.argmax(norms)), int(np.argmin(norms))
    assert norms[big] / norms[small] > 5.0  # sigma = 1 over 64 draws spreads far wider
    check = [3 * big, 3 * big + 1, 3 * big + 2, 3 * small, 3 * small + 1, 3 * small + 2, 192]
    rng = np.random.default_rng(5)
    sample = rng.integers(0, N, 2_000_000)
    # plus every element of the checked matrices
    sample = np.unique(np.concatenate([sample] + [np.arange(offs[i], offs[i + 1]) for i in check]))
    # the checks hold for both extremes: the kernels' normalisation (scale invariance of
    # the iteration) makes O independent of each expert's gradient scale
    reps = _step_and_check(capi, wl, W0, G0, check, sample=sample)
    assert len(reps) == 7

"""GPU parity at full size: the Llama-3-8B matrix set (224 matrices, 6.98e9 elements per
fp32 buffer) in the launch configuration bench.py times, and its 8-shard variant with
straddling parameters (bf16, fp32 and split-fp32 Newton-Schulz).

The oracle cannot run the whole step, so the checks are (a) bit-exact gather / scatter
over every element, (b) momentum and weights on a seeded sample of a million flat
positions, computed one by one in fp64 and bounded element by element, and (c)
Newton-Schulz on sampled matrices of each kind (wide k/v, square q/o, tall gate/up, wide
down), run by the oracle on the GPU's own stored input and bounded whole, per 128 x 128
tile and per element (tests/parity.py).  One test runs muon_step itself, the fused path
bench.py times, with the default kernel choice.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle import muon_ref as ref  # noqa: E402
from muon_optimizer_step_gb300 import inputs  # noqa: E402
from tests import parity  # noqa: E402

TOL_NS = {0: 2e-2, 1: 1e-4, 2: 1e-4}
TOL_STATE = 1e-6
LAYER = 7  # q, o, k, v, gate, up, down


@pytest.fixture(scope="module")
def capi():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, total = torch.cuda.mem_get_info()
    if free < 200e9:
        pytest.skip("needs ~200 GB of free device memory")
    from muon_optimizer_step_gb300 import capi as c
    return c


def rel(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    return float(np.linalg.norm(x - y) / np.linalg.norm(y))


def run_full(capi, wl_name, ns_dtype, sample_params):
    wl = inputs.WORKLOADS[wl_name]
    lay = capi.muon_layout_create(wl.shapes, wl.n_shards, ns_dtype, wl.is_matrix)
    S, L, N = wl.n_shards, lay.shard_len, lay.numel
    Wb = torch.zeros(S * L, device="cuda")
    Gb = torch.zeros(S * L, device="cuda")
    Mb = torch.zeros(S * L, device="cuda")
    inputs.device_fill_weights(wl, Wb[:N])
    inputs.device_fill_grads(wl, Gb[:N], 0)
    W = [Wb[s * L:(s + 1) * L] for s in range(S)]
    G = [Gb[s * L:(s + 1) * L] for s in range(S)]
    M = [Mb[s * L:(s + 1) * L] for s in range(S)]
    ws = capi.workspace_tensor(lay)
    rng = np.random.default_rng(123)
    mat_pos = []
    pos = 0
    for i, (r, c) in enumerate(wl.shapes):
        if wl.is_matrix[i]:
            mat_pos.append((pos, pos + r * c))
        pos += r * c
    # a million sampled flat positions inside matrices
    starts = np.array([a for a, _ in mat_pos])
    sizes = np.array([b - a for a, b in mat_pos])
    pick = rng.choice(len(mat_pos), 1_000_000, p=sizes / sizes.sum())
    idx = torch.from_numpy(starts[pick] + (rng.random(1_000_000) * sizes[pick]).astype(np.int64)).cuda()
    W_prev = Wb[idx].double().cpu().numpy()
    G_s = Gb[idx].double().cpu().numpy()
    # ---- full gather is a bit-exact copy of every matrix element
    full = torch.empty(lay.full_numel, device="cuda")
    capi.muon_gather_full(lay, W, full)
    torch.cuda.synchronize()
    for i, (r, c) in enumerate(wl.shapes):
        if wl.is_matrix[i]:
            off = lay.full_offsets[i]
            fo = int(np.sum([a * b for a, b in wl.shapes[:i]]))
            assert torch.equal(full[off: off + r * c], Wb[fo: fo + r * c]), i
    # ---- scatter of the same values back into zeroed shards restores the matrix positions
    Z = torch.zeros(S * L, device="cuda")
    capi.muon_scatter_updates(lay, full, [Z[s * L:(s + 1) * L] for s in range(S)])
    torch.cuda.synchronize()
    prev = 0
    for a, b in mat_pos:  # views only: no copies of the 28 GB buffers
        assert torch.equal(Z[a:b], Wb[a:b])
        if a > prev:
            assert not Z[prev:a].any()
        prev = b
    assert not Z[prev:].any()
    del Z
    # ---- the step, stage by stage
    capi.muon_compute_momentum_inputs(G, M, lay, ws, wl.mu, wl.nesterov)
    capi.muon_export_input(lay, ws, full)
    torch.cuda.synchronize()
    X_in = {}
    for i in sample_params:
        r, c = wl.shapes[i]
        off = lay.full_offsets[i]
        X_in[i] = full[off: off + r * c].view(r, c).double().cpu().numpy()
    capi.muon_orthogonalize_updates(lay, ws, wl.ns_steps)
    capi.muon_export_update(lay, ws, wl.ns_steps, full)
    capi.muon_apply_local_updates(W, lay, ws, wl.lr, wl.wd, wl.ns_steps)
    capi.muon_check()
    # momentum on the sample (M0 = 0): M1 = G
    M_s = Mb[idx].double().cpu().numpy()
    assert rel(M_s, ref.momentum_update(np.zeros_like(G_s), G_s, wl.mu)) < TOL_STATE
    parity.check_momentum(M_s, ref.momentum_update(np.zeros_like(G_s), G_s, wl.mu), 0.0, "sample")
    # weights on the sample, given the GPU's own O
    flat_to_full = np.zeros(len(wl.shapes), dtype=np.int64)
    for i in range(len(wl.shapes)):
        flat_to_full[i] = lay.full_offsets[i] - int(np.sum([a * b for a, b in wl.shapes[:i]])) \
            if wl.is_matrix[i] else 0
    owner = np.searchsorted(np.cumsum([r * c for r, c in wl.shapes]), idx.cpu().numpy(), side="right")
    O_s = full[torch.from_numpy(idx.cpu().numpy() + flat_to_full[owner]).cuda()].double().cpu().numpy()
    scale = np.array([ref.update_scale(*wl.shapes[k]) for k in owner])
    want_w = ref.weight_decay(W_prev, wl.lr, wl.wd) - wl.lr * scale * O_s
    W_s = Wb[idx].double().cpu().numpy()
    assert rel(W_s, want_w) < TOL_STATE
    parity.check_weights(W_s, want_w, W_prev, 1 - wl.lr * wl.wd, wl.lr * scale * O_s, what="sample")
    # Newton-Schulz on sampled matrices, oracle on the GPU's stored input
    for i in sample_params:
        r, c = wl.shapes[i]
        off = lay.full_offsets[i]
        O = full[off: off + r * c].view(r, c).double().cpu().numpy()
        rep = parity.check_ns(O, ref.newton_schulz(X_in[i], wl.ns_steps), ns_dtype, (i, (r, c)))
        print("NS", wl_name, ns_dtype, i, (r, c), rep)
    del Wb, Gb, Mb, W, G, M, ws, full
    torch.cuda.empty_cache()


def test_llama_full_size_bf16(capi):
    # layer 0 k (wide 1024x4096), layer 5 q (square), layer 31 gate (tall 14336x4096),
    # layer 17 down (wide 4096x14336)
    run_full(capi, "llama3_8b_x32", 0, [0 * LAYER + 2, 5 * LAYER + 0, 31 * LAYER + 4,
                                        17 * LAYER + 6])


def test_llama_8_shards_straddling_bf16(capi):
    # index 0 is the leading vector; layer 3's down projection straddles shards 0 and 1
    run_full(capi, "llama3_8b_8shards", 0, [1 + 3 * LAYER + 3, 1 + 3 * LAYER + 6])


def test_llama_8_shards_fp32_ns(capi):
    run_full(capi, "llama3_8b_8shards", 1, [1 + 0 * LAYER + 2, 1 + 9 * LAYER + 1])


def test_llama_8_shards_split_fp32_ns(capi):
    # layer 2's gate (tall: MN-major Gram operands), layer 3's down projection (wide,
    # straddling shards 0 and 1: MN-major Update operand)
    run_full(capi, "llama3_8b_8shards", 2, [1 + 2 * LAYER + 4, 1 + 3 * LAYER + 6])


def test_llama_full_size_muon_step_fused(capi):
    """muon_step itself on the 32-layer set: the default kernel choice (as bench.py runs
    it), momentum and inputs on the GPU, Newton-Schulz, and the last Update applying W in
    its epilogue.  Checked:
      * momentum on a million sampled positions (M0 = 0, so M1 = G exactly);
      * the update O (the bf16 values the last Update stores) of one matrix of every shape
        against the oracle's Newton-Schulz of the GPU's own input, which is rebuilt on the
        host bit for bit: X = bf16(fp32(0.95f * G + G)) (with M0 = 0 the Nesterov input
        is one fp32 fused multiply-add of G, then rounded to bf16);
      * W on the sample against the oracle's decay and apply of that O, within the bf16
        rounding of O (the fused tail applies the fp32 value before rounding it):
        lr * s * 2^-8 * |O| per element, plus the fp32 floor."""
    wl = inputs.WORKLOADS["llama3_8b_x32"]
    lay = capi.muon_layout_create(wl.shapes, 1, 0, wl.is_matrix)
    k = capi.muon_layout_ns_kernel(lay)
    N = lay.numel
    W = torch.zeros(N, device="cuda")
    G = torch.zeros(N, device="cuda")
    M = torch.zeros(N, device="cuda")
    inputs.device_fill_weights(wl, W)
    inputs.device_fill_grads(wl, G, 0)
    ws = capi.workspace_tensor(lay)
    rng = np.random.default_rng(321)
    idx = torch.from_numpy(rng.integers(0, N, 1_000_000)).cuda()
    W_prev = W[idx].double().cpu().numpy()
    pick = [0 * LAYER + 0, 3 * LAYER + 3, 30 * LAYER + 5, 31 * LAYER + 6]  # q, v, up, down
    offs = np.concatenate([[0], np.cumsum([r * c for r, c in wl.shapes])])
    G_m = {i: G[offs[i]: offs[i + 1]].cpu().numpy() for i in pick}
    torch.cuda.synchronize()
    capi.muon_step([W], [G], [M], lay, ws, wl.lr, wl.wd, wl.mu, wl.nesterov, wl.ns_steps)
    full = torch.empty(lay.full_numel, device="cuda")
    capi.muon_export_update(lay, ws, wl.ns_steps, full)
    capi.muon_check()
    G_s = G[idx].double().cpu().numpy()
    parity.check_momentum(M[idx].double().cpu().numpy(),
                          ref.momentum_update(np.zeros_like(G_s), G_s, wl.mu), 0.0, "sample")
    del M
    # every sampled position lies in some matrix (the set has no vectors)
    owner = np.searchsorted(offs[1:], idx.cpu().numpy(), side="right")
    pos_full = np.array(lay.full_offsets)[owner] + (idx.cpu().numpy() - offs[owner])
    O_s = full[torch.from_numpy(pos_full).cuda()].double().cpu().numpy()
    scale = np.array([ref.update_scale(*wl.shapes[j]) for j in owner])
    want_w = ref.weight_decay(W_prev, wl.lr, wl.wd) - wl.lr * scale * O_s
    lrs_o = wl.lr * scale * O_s
    parity.check_weights(W[idx].double().cpu().numpy(), want_w, W_prev, 1 - wl.lr * wl.wd, lrs_o,
                         extra=parity.BF16_REL * np.abs(lrs_o), what=("fused tail", k))
    mu32 = np.float64(np.float32(wl.mu))
    for i in pick:
        r, c = wl.shapes[i]
        g = G_m[i].astype(np.float64)
        X = parity.bf16_round((mu32 * g + g).astype(np.float32)).astype(np.float64).reshape(r, c)
        off = lay.full_offsets[i]
        O = full[off: off + r * c].view(r, c).double().cpu().numpy()
        rep = parity.check_ns(O, ref.newton_schulz(X, wl.ns_steps), 0, (i, (r, c), k))
        print("NS fused", i, (r, c), k, rep)
    del W, G, ws, full
    torch.cuda.empty_cache()

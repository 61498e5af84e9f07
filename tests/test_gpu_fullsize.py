"""GPU parity at full size: the Llama-3-8B matrix set (224 matrices, 6.98e9 elements per
fp32 buffer) in the launch configuration bench.py times, and its 8-shard variant with
straddling parameters (bf16, fp32 and split-fp32 Newton-Schulz).

The oracle cannot run the whole step, so the checks are (a) bit-exact gather / scatter
over every element, (b) momentum and weights on a seeded sample of a million flat
positions, computed one by one in fp64, and (c) Newton-Schulz on sampled matrices of
each kind (wide k/v, square q/o, tall gate/up), run by the oracle on the GPU's own
stored input.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle import muon_ref as ref  # noqa: E402
from muon_optimizer_step_gb300 import inputs  # noqa: E402

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
    # weights on the sample, given the GPU's own O
    flat_to_full = np.zeros(len(wl.shapes), dtype=np.int64)
    for i in range(len(wl.shapes)):
        flat_to_full[i] = lay.full_offsets[i] - int(np.sum([a * b for a, b in wl.shapes[:i]])) \
            if wl.is_matrix[i] else 0
    owner = np.searchsorted(np.cumsum([r * c for r, c in wl.shapes]), idx.cpu().numpy(), side="right")
    O_s = full[torch.from_numpy(idx.cpu().numpy() + flat_to_full[owner]).cuda()].double().cpu().numpy()
    scale = np.array([ref.update_scale(*wl.shapes[k]) for k in owner])
    want_w = ref.weight_decay(W_prev, wl.lr, wl.wd) - wl.lr * scale * O_s
    assert rel(Wb[idx].double().cpu().numpy(), want_w) < TOL_STATE
    # Newton-Schulz on sampled matrices, oracle on the GPU's stored input
    for i in sample_params:
        r, c = wl.shapes[i]
        off = lay.full_offsets[i]
        O = full[off: off + r * c].view(r, c).double().cpu().numpy()
        e = rel(O, ref.newton_schulz(X_in[i], wl.ns_steps))
        assert e < TOL_NS[ns_dtype], (i, (r, c), e)
    del Wb, Gb, Mb, W, G, M, ws, full
    torch.cuda.empty_cache()


def test_llama_full_size_bf16(capi):
    # layer 0 k (wide 1024x4096), layer 5 q (square), layer 31 gate (tall 14336x4096)
    run_full(capi, "llama3_8b_x32", 0, [0 * LAYER + 2, 5 * LAYER + 0, 31 * LAYER + 4])


def test_llama_8_shards_straddling_bf16(capi):
    # index 0 is the leading vector; layer 3's down projection straddles shards 0 and 1
    run_full(capi, "llama3_8b_8shards", 0, [1 + 3 * LAYER + 3, 1 + 3 * LAYER + 6])


def test_llama_8_shards_fp32_ns(capi):
    run_full(capi, "llama3_8b_8shards", 1, [1 + 0 * LAYER + 2, 1 + 9 * LAYER + 1])


def test_llama_8_shards_split_fp32_ns(capi):
    # layer 2's gate (tall: MN-major Gram operands), layer 3's down projection (wide,
    # straddling shards 0 and 1: MN-major Update operand)
    run_full(capi, "llama3_8b_8shards", 2, [1 + 2 * LAYER + 4, 1 + 3 * LAYER + 6])

"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, stage by stage.

Every Newton-Schulz output is checked whole, per 128 x 128 tile and per element, and the
momentum, input and weights element by element (tests/parity.py states the bounds).
Tolerances (relative Frobenius error ||gpu - oracle|| / ||oracle||, per matrix):
  * gather / scatter, non-matrix bytes, shard padding: bit-exact;
  * momentum M and weights W: 1e-6 (fp32 arithmetic, one or two roundings per element);
  * stored orthogonalization input X: 2e-3 on the bf16 path (round-to-nearest bf16 has
    relative error <= 2^-9 per element), 1e-6 on the fp32 and split-fp32 paths (the latter
    keeps h + m + l, within 2^-26 of each value);
  * Newton-Schulz output: 2e-2 on the bf16 path, 1e-4 on the fp32 and split-fp32 paths, both
    against the oracle run on the GPU's own stored input and against the oracle's own
    input.
W is compared as oracle_apply(W_before, O_gpu) against W_gpu, so the NS tolerance does not
leak into the 1e-6 weight check.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle import muon_ref as ref  # noqa: E402
from muon_optimizer_step_gb300 import inputs  # noqa: E402
from tests import parity  # noqa: E402

TOL_NS = {0: 2e-2, 1: 1e-4, 2: 1e-4}
TOL_X = {0: 2e-3, 1: 1e-6, 2: 1e-6}
TOL_STATE = 1e-6


@pytest.fixture(scope="module")
def capi():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from muon_optimizer_step_gb300 import capi as c
    return c


def rel(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    d = np.linalg.norm(y)
    return float(np.linalg.norm(x - y) / d) if d > 0 else float(np.linalg.norm(x))


def split_shards(flat, n_shards):
    """Plain numpy split of a flat vector into n_shards zero-padded shards of ceil(N/S)."""
    flat = np.asarray(flat, dtype=np.float32)
    L = -(-flat.size // n_shards)
    padded = np.zeros(L * n_shards, dtype=np.float32)
    padded[: flat.size] = flat
    return [torch.from_numpy(padded[s * L:(s + 1) * L].copy()).cuda() for s in range(n_shards)]


def join_shards(shards, N):
    return np.concatenate([s.cpu().numpy() for s in shards])[:N]


def full_to_mats(full, layout, wl):
    full = full.cpu().numpy() if hasattr(full, "cpu") else full
    out = {}
    for i, (r, c) in enumerate(wl.shapes):
        if wl.is_matrix[i]:
            off = layout.full_offsets[i]
            out[i] = full[off: off + r * c].reshape(r, c).astype(np.float64)
    return out


def mats_to_full(mats, layout):
    full = np.zeros(max(1, layout.full_numel), dtype=np.float32)
    for i, X in mats.items():
        off = layout.full_offsets[i]
        full[off: off + X.size] = np.asarray(X, dtype=np.float32).reshape(-1)
    return torch.from_numpy(full).cuda()


def matrix_mask(wl, N):
    mask = np.zeros(N, dtype=bool)
    pos = 0
    for i, (r, c) in enumerate(wl.shapes):
        if wl.is_matrix[i]:
            mask[pos:pos + r * c] = True
        pos += r * c
    return mask


# ------------------------------------------------------------------ gather / scatter
@pytest.mark.parametrize("n_shards", [1, 3, 8])
def test_gather_scatter_bit_exact(capi, n_shards):
    wl = inputs.WORKLOADS["ragged_small"]
    lay = capi.muon_layout_create(wl.shapes, n_shards, 0, wl.is_matrix)
    N = lay.numel
    rng = np.random.default_rng(n_shards)
    flat = rng.normal(size=N).astype(np.float32)
    shards = split_shards(flat, n_shards)
    full = torch.full((lay.full_numel,), float("nan"), device="cuda")
    capi.muon_gather_full(lay, shards, full)
    torch.cuda.synchronize()
    o = ref.flat_layout(wl.shapes, n_shards, wl.is_matrix)
    want = ref.gather_full(ref.shard_flat(flat, o), o)
    got = full_to_mats(full, lay, wl)
    for i in want:
        assert np.array_equal(got[i].astype(np.float32), want[i].astype(np.float32)), i
    # scatter of fresh values into sentinel shards touches matrix positions only
    y = {i: rng.normal(size=want[i].shape).astype(np.float32) for i in want}
    sent = split_shards(np.full(N, 7.0, dtype=np.float32), n_shards)
    for s in sent:
        s.fill_(7.0)
    capi.muon_scatter_updates(lay, mats_to_full(y, lay), sent)
    torch.cuda.synchronize()
    back = np.concatenate([s.cpu().numpy() for s in sent])
    want_sh = ref.scatter_updates(y, o, [np.full(o["L"], 7.0) for _ in range(n_shards)])
    assert np.array_equal(back, np.concatenate(want_sh).astype(np.float32))


@pytest.mark.parametrize("n_shards,seed", [(2, 1), (7, 2), (128, 3)])
def test_gather_scatter_random_layouts(capi, n_shards, seed):
    """Gather and scatter bit-exact against the oracle's index maps on random shapes
    (vectors mixed in, so matrices straddle shard edges at random places), up to the
    largest shard count."""
    rng = np.random.default_rng(seed)
    shapes = [(int(rng.integers(1, 300)), int(rng.integers(1, 300))) for _ in range(12)]
    is_matrix = [bool(rng.random() < 0.8) for _ in shapes]
    lay = capi.muon_layout_create(shapes, n_shards, 0, is_matrix)
    N = lay.numel
    flat = rng.normal(size=N).astype(np.float32)
    full = torch.full((max(1, lay.full_numel),), float("nan"), device="cuda")
    capi.muon_gather_full(lay, split_shards(flat, n_shards), full)
    torch.cuda.synchronize()
    o = ref.flat_layout(shapes, n_shards, is_matrix)
    want = ref.gather_full(ref.shard_flat(flat, o), o)
    f = full.cpu().numpy()
    for i, (r, c) in enumerate(shapes):
        if is_matrix[i]:
            off = lay.full_offsets[i]
            assert np.array_equal(f[off: off + r * c].reshape(r, c), want[i].astype(np.float32)), i
    y = {i: rng.normal(size=want[i].shape).astype(np.float32) for i in want}
    sent = split_shards(np.full(N, 5.0, dtype=np.float32), n_shards)
    for t in sent:
        t.fill_(5.0)
    capi.muon_scatter_updates(lay, mats_to_full(y, lay), sent)
    torch.cuda.synchronize()
    back = np.concatenate([t.cpu().numpy() for t in sent])
    want_sh = ref.scatter_updates(y, o, [np.full(o["L"], 5.0) for _ in range(n_shards)])
    assert np.array_equal(back, np.concatenate(want_sh).astype(np.float32))


# ------------------------------------------------------------------ Newton-Schulz on given inputs
def spectrum_inputs(wl, seed):
    rng = np.random.default_rng(seed)
    mats = {}
    for i, (r, c) in enumerate(wl.shapes):
        if not wl.is_matrix[i]:
            continue
        k = min(r, c)
        U, _ = np.linalg.qr(rng.normal(size=(r, k)))
        V, _ = np.linalg.qr(rng.normal(size=(c, k)))
        s = np.exp(rng.uniform(np.log(1e-3), 0.0, size=k))  # three decades of spectrum
        mats[i] = (U * s) @ V.T * rng.uniform(1e-3, 10.0)
    return mats


def recipe_inputs(wl, seed):
    """Gradient-like inputs (the workload recipe: noise plus low-rank), each matrix scaled
    by a random factor in [1e-3, 10] (the iteration is scale invariant)."""
    rng = np.random.default_rng(seed)
    g = inputs.host_grads(wl, seed)
    mats = {}
    pos = 0
    for i, (r, c) in enumerate(wl.shapes):
        if wl.is_matrix[i]:
            mats[i] = g[pos:pos + r * c].reshape(r, c).astype(np.float64) * rng.uniform(1e-3, 10.0)
        pos += r * c
    return mats


# The 2e-2 bound of the bf16 path holds for gradient-like inputs; with singular values
# spread over three decades, bf16 rounding of X, A and B alone (emulated on the CPU)
# gives 4e-2 to 1e-1, so that family is checked on the fp32 path only.
@pytest.mark.parametrize("ns_dtype,family", [(0, "recipe"), (1, "recipe"), (1, "spectrum"),
                                             (2, "recipe"), (2, "spectrum")])
@pytest.mark.parametrize("ns_steps", [5, 1, 0])
def test_orthogonalize_full_vs_oracle(capi, ns_dtype, family, ns_steps):
    wl = inputs.WORKLOADS["ragged_small"]
    lay = capi.muon_layout_create(wl.shapes, 1, ns_dtype, wl.is_matrix)
    ws = capi.workspace_tensor(lay)
    X = (recipe_inputs if family == "recipe" else spectrum_inputs)(wl, 10 + ns_steps)
    out = torch.zeros(lay.full_numel, device="cuda")
    capi.muon_orthogonalize_full(lay, ws, mats_to_full(X, lay), out, ns_steps)
    capi.muon_check()
    got = full_to_mats(out, lay, wl)
    for i, Xi in X.items():
        want = ref.newton_schulz(Xi.astype(np.float32).astype(np.float64), ns_steps)
        assert got[i].shape == want.shape
        parity.check_ns(got[i], want, ns_dtype, (i, wl.shapes[i]))


@pytest.mark.parametrize("ns_dtype", [0, 1, 2])
def test_orthogonalize_zero_matrix_gives_zero(capi, ns_dtype):
    shapes = [(130, 300), (5, 5)]
    lay = capi.muon_layout_create(shapes, 1, ns_dtype)
    ws = capi.workspace_tensor(lay)
    rng = np.random.default_rng(0)
    Q, _ = np.linalg.qr(rng.normal(size=(5, 5)))
    R, _ = np.linalg.qr(rng.normal(size=(5, 5)))
    X5 = (Q @ np.diag([3.0, 2.5, 2.0, 1.5, 1.0]) @ R.T).astype(np.float32)
    fin = torch.zeros(lay.full_numel, device="cuda")
    off = lay.full_offsets[1]
    fin[off: off + 25] = torch.from_numpy(X5.reshape(-1)).cuda()
    out = torch.full((lay.full_numel,), float("nan"), device="cuda")
    capi.muon_orthogonalize_full(lay, ws, fin, out, 5)
    capi.muon_check()
    o = out.cpu().numpy()
    assert np.all(o[:130 * 300] == 0.0)
    want = ref.newton_schulz(X5.astype(np.float64))
    parity.check_ns(o[off:off + 25].reshape(5, 5), want, ns_dtype, "5x5 beside a zero matrix")


# ------------------------------------------------------------------ the step, stage by stage
def run_steps(capi, wl, n_shards, ns_dtype, n_steps, check):
    lay = capi.muon_layout_create(wl.shapes, n_shards, ns_dtype, wl.is_matrix)
    ws = capi.workspace_tensor(lay)
    N = lay.numel
    W0, Gs, M0 = inputs.host_inputs(wl)
    W = split_shards(W0, n_shards)
    M = split_shards(M0, n_shards)
    mask = matrix_mask(wl, N)
    o = ref.flat_layout(wl.shapes, n_shards, wl.is_matrix)
    fin = torch.zeros(max(1, lay.full_numel), device="cuda")
    fout = torch.zeros(max(1, lay.full_numel), device="cuda")
    M_or = M0.astype(np.float64)
    for t in range(n_steps):
        G = split_shards(Gs[t], n_shards)
        W_prev = join_shards(W, N)
        M_prev = join_shards(M, N)
        capi.muon_compute_momentum_inputs(G, M, lay, ws, wl.mu, wl.nesterov)
        capi.muon_export_input(lay, ws, fin)
        capi.muon_orthogonalize_updates(lay, ws, wl.ns_steps)
        capi.muon_export_update(lay, ws, wl.ns_steps, fout)
        capi.muon_apply_local_updates(W, lay, ws, wl.lr, wl.wd, wl.ns_steps)
        capi.muon_check()
        W_new = join_shards(W, N)
        M_new = join_shards(M, N)
        # momentum, against the oracle's own running momentum (M never depends on W or O),
        # and element by element against the oracle's step from the GPU's previous M
        M_or = np.where(mask, ref.momentum_update(M_or, Gs[t], wl.mu), M_or)
        assert rel(M_new[mask], M_or[mask]) < TOL_STATE
        M_stage = ref.momentum_update(M_prev, Gs[t], wl.mu)
        parity.check_momentum(M_new[mask], M_stage[mask], wl.mu * M_prev[mask].astype(np.float64),
                              ("step", t))
        assert np.array_equal(M_new[~mask], M_prev[~mask])
        X_gpu = full_to_mats(fin, lay, wl)
        O_gpu = full_to_mats(fout, lay, wl)
        X_or = ref.gather_full(ref.shard_flat(ref.ns_input(Gs[t], M_or, wl.mu, wl.nesterov), o), o)
        X_stage = ref.gather_full(ref.shard_flat(ref.ns_input(Gs[t], M_stage, wl.mu, wl.nesterov),
                                                 o), o)
        G_full = ref.gather_full(ref.shard_flat(Gs[t], o), o)
        for i in X_or:
            r, c = wl.shapes[i]
            assert rel(X_gpu[i], X_or[i]) < TOL_X[ns_dtype], ("X", i)
            parity.check_input(X_gpu[i], X_stage[i], G_full[i], ns_dtype, ("X", i))
            parity.check_ns(O_gpu[i], ref.newton_schulz(X_gpu[i], wl.ns_steps), ns_dtype, ("O", i))
            assert rel(O_gpu[i], ref.newton_schulz(X_or[i], wl.ns_steps)) < TOL_NS[ns_dtype], ("O*", i)
            off = o["offsets"][i]
            Wp = W_prev[off: off + r * c].astype(np.float64)
            want = ref.apply_update(ref.weight_decay(Wp, wl.lr, wl.wd), O_gpu[i].reshape(-1), wl.lr,
                                    r, c)
            assert rel(W_new[off: off + r * c], want) < TOL_STATE, ("W", i)
            lrs_o = wl.lr * ref.update_scale(r, c) * O_gpu[i].reshape(-1)
            parity.check_weights(W_new[off: off + r * c], want, Wp, 1 - wl.lr * wl.wd, lrs_o,
                                 what=("W", i))
        assert np.array_equal(W_new[~mask], W_prev[~mask])
        # shard padding never touched
        pad = np.concatenate([s.cpu().numpy() for s in W])[N:]
        assert not pad.any()
        if check is not None:
            check(t, W, M)
    return lay, W, M


@pytest.mark.parametrize("ns_dtype", [0, 1, 2])
def test_single_256x128_three_steps(capi, ns_dtype):
    run_steps(capi, inputs.WORKLOADS["single_256x128"], 1, ns_dtype, 3, None)


@pytest.mark.parametrize("ns_dtype", [0, 1, 2])
@pytest.mark.parametrize("n_shards", [1, 3])
def test_ragged_two_steps(capi, ns_dtype, n_shards):
    run_steps(capi, inputs.WORKLOADS["ragged_small"], n_shards, ns_dtype, 2, None)


@pytest.mark.parametrize("ns_dtype", [0, 1, 2])
def test_step_equals_stages_and_sharding_is_exact(capi, ns_dtype):
    """muon_step = stage 1 + muon_orthogonalize_apply, bit for bit; 1 vs 5 shards bit for
    bit; and against the three separate stages: equal on the fp32 path, and on the bf16
    path (whose fused tail applies the fp32 O instead of its bf16 rounding) within the
    rounding of two steps' O (bf16 keeps 8 significant bits, so each element of O is off by
    at most 2^-8 of itself): sum_t lr * scale * 2^-8 * ||O_t|| ~ lr * scale * 2^-7 * ||O_2||
    (the two steps' updates have nearly equal norms)."""
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    results = []
    O_last = None
    for n_shards, mode in [(1, "step"), (5, "step"), (5, "fused"), (5, "stages")]:
        lay = capi.muon_layout_create(wl.shapes, n_shards, ns_dtype, wl.is_matrix)
        ws = capi.workspace_tensor(lay)
        W = split_shards(W0, n_shards)
        M = split_shards(M0, n_shards)
        for t in range(2):
            G = split_shards(Gs[t], n_shards)
            if mode == "step":
                capi.muon_step(W, G, M, lay, ws, wl.lr, wl.wd, wl.mu, True, 5)
            else:
                capi.muon_compute_momentum_inputs(G, M, lay, ws, wl.mu, True)
                if mode == "fused":
                    capi.muon_orthogonalize_apply(W, lay, ws, wl.lr, wl.wd, 5)
                else:
                    capi.muon_orthogonalize_updates(lay, ws, 5)
                    capi.muon_apply_local_updates(W, lay, ws, wl.lr, wl.wd, 5)
        if mode == "stages":
            O_last = torch.zeros(lay.full_numel, device="cuda")
            capi.muon_export_update(lay, ws, 5, O_last)
        capi.muon_check()
        results.append((join_shards(W, lay.numel), join_shards(M, lay.numel)))
    for Wr, Mr in results[1:3]:
        assert np.array_equal(Wr, results[0][0])
        assert np.array_equal(Mr, results[0][1])
    W_st, M_st = results[3]
    assert np.array_equal(M_st, results[0][1])
    if ns_dtype == 1:
        assert np.array_equal(W_st, results[0][0])
        return
    o = ref.flat_layout(wl.shapes, 1, wl.is_matrix)
    O = full_to_mats(O_last, capi.muon_layout_create(wl.shapes, 1, 0, wl.is_matrix), wl)
    # per step, the staged apply reads O rounded to bf16 (2^-8 of each element) or, on
    # the split-fp32 path, as h + m + l (2^-26)
    factor = 2.0 ** -7 if ns_dtype == 0 else 2.0 ** -20
    for i, Oi in O.items():
        r, c = wl.shapes[i]
        sl = slice(o["offsets"][i], o["offsets"][i] + r * c)
        bound = wl.lr * ref.update_scale(r, c) * factor * np.linalg.norm(Oi) \
            + 1e-6 * np.linalg.norm(W_st[sl].astype(np.float64))
        diff = np.linalg.norm(results[0][0][sl].astype(np.float64) - W_st[sl])
        assert diff <= bound, (i, diff, bound)


def test_repeat_runs_are_bit_identical(capi):
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    outs = []
    for _ in range(2):
        lay = capi.muon_layout_create(wl.shapes, 2, 0, wl.is_matrix)
        ws = capi.workspace_tensor(lay)
        W, M, G = split_shards(W0, 2), split_shards(M0, 2), split_shards(Gs[0], 2)
        capi.muon_step(W, G, M, lay, ws, wl.lr, wl.wd, wl.mu, True, 5)
        capi.muon_check()
        outs.append(join_shards(W, lay.numel))
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("nesterov", [True, False])
def test_plain_momentum_and_zero_ns_steps(capi, nesterov):
    wl = inputs.WORKLOADS["single_256x128"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    lay = capi.muon_layout_create(wl.shapes, 1, 1)
    ws = capi.workspace_tensor(lay)
    W, M, G = split_shards(W0, 1), split_shards(M0 + 0.5, 1), split_shards(Gs[0], 1)
    capi.muon_step(W, G, M, lay, ws, wl.lr, wl.wd, wl.mu, nesterov, 0)
    capi.muon_check()
    Mo = ref.momentum_update(M0 + 0.5, Gs[0], wl.mu)
    X = ref.ns_input(Gs[0], Mo, wl.mu, nesterov).reshape(256, 128)
    O = ref.newton_schulz(X, 0)  # X / ||X||
    want = ref.apply_update(ref.weight_decay(W0, wl.lr, wl.wd), O.reshape(-1), wl.lr, 256, 128)
    assert rel(join_shards(M, lay.numel), Mo) < TOL_STATE
    assert rel(join_shards(W, lay.numel), want) < 2e-6


def test_empty_layout_is_a_noop(capi):
    lay = capi.muon_layout_create([(4, 1)], 1, 0, [False])
    ws = capi.workspace_tensor(lay)
    W = torch.arange(4, dtype=torch.float32, device="cuda")
    M = torch.ones(4, device="cuda")
    G = torch.ones(4, device="cuda")
    capi.muon_step([W], [G], [M], lay, ws, 0.02, 0.01, 0.95, True, 5)
    capi.muon_check()
    assert torch.equal(W.cpu(), torch.arange(4, dtype=torch.float32))
    assert torch.equal(M.cpu(), torch.ones(4))


def test_wait_timeout_is_reported_and_context_survives(capi):
    capi.muon_check()  # clean slate
    capi.muon_selftest_wait_timeout(1_000_000)
    assert capi.muon_check_status() == capi.MUON_ERR_TIMEOUT
    assert capi.muon_check_status() == capi.MUON_OK  # cleared
    x = torch.ones(8, device="cuda") * 2
    assert float(x.sum()) == 16.0


@pytest.mark.parametrize("variant", ["1", "2", "3"])
@pytest.mark.parametrize("persistent", ["0", "1"])
def test_each_tcgen05_variant_vs_oracle(capi, variant, persistent, monkeypatch):
    """The three tcgen05 tile shapes (single CTA 128x256 tiles; 256x256 and 256x512 tiles
    on CTA pairs) and both launch modes (one launch per phase; one persistent launch whose tiles wait on
    per-matrix counters), pinned one at a time, on ragged shapes and on a matrix that
    spans several pair tiles."""
    monkeypatch.setenv("MUON_TC_KERNEL", variant)
    monkeypatch.setenv("MUON_NS_PERSISTENT", persistent)
    shapes = [(300, 200), (130, 520), (7, 3), (64, 1000), (257, 129), (600, 1100), (1100, 600)]
    wl = inputs.Workload("mixed", tuple(shapes), (True,) * len(shapes), 1, seed=9, rank=4)
    lay = capi.muon_layout_create(wl.shapes, 1, 0, wl.is_matrix)
    k = capi.muon_layout_ns_kernel(lay)
    assert k["tile_shape"] == int(variant) and k["persistent"] == (persistent == "1"), k
    assert k["units"] >= 1
    ws = capi.workspace_tensor(lay)
    X = recipe_inputs(wl, 3)
    out = torch.zeros(lay.full_numel, device="cuda")
    capi.muon_orthogonalize_full(lay, ws, mats_to_full(X, lay), out, 5)
    capi.muon_check()
    got = full_to_mats(out, lay, wl)
    for i, Xi in X.items():
        parity.check_ns(got[i], ref.newton_schulz(Xi.astype(np.float32).astype(np.float64), 5), 0,
                        (variant, persistent, wl.shapes[i]))


@pytest.mark.parametrize("variant", ["1", "2", "3"])
def test_persistent_lists_past_the_planned_iterations(capi, variant, monkeypatch):
    """A persistent launch plans tile lists for six iterations and reuses the sixth's for
    later ones.  Each tile computes the same bits whichever list holds it, so the
    persistent launch must equal one launch per phase bit for bit, here at 8 iterations
    (and at 6 and 1, the planned and the shortest case)."""
    monkeypatch.setenv("MUON_TC_KERNEL", variant)
    shapes = [(300, 200), (130, 520), (7, 3), (64, 1000), (257, 129), (600, 1100), (1100, 600),
              (768, 768), (768, 2304)]
    wl = inputs.Workload("mixed_long", tuple(shapes), (True,) * len(shapes), 1, seed=12, rank=4)
    X = recipe_inputs(wl, 4)
    lays = {}
    for pers in ("1", "0"):
        monkeypatch.setenv("MUON_NS_PERSISTENT", pers)
        lay = capi.muon_layout_create(wl.shapes, 1, 0, wl.is_matrix)
        assert capi.muon_layout_ns_kernel(lay)["persistent"] == (pers == "1")
        lays[pers] = lay
    for ns_steps in (8, 6, 1):
        outs = {}
        for pers, lay in lays.items():
            ws = capi.workspace_tensor(lay)
            out = torch.zeros(lay.full_numel, device="cuda")
            capi.muon_orthogonalize_full(lay, ws, mats_to_full(X, lay), out, ns_steps)
            capi.muon_check()
            outs[pers] = out.cpu()
        assert torch.equal(outs["1"], outs["0"]), (variant, ns_steps)
        assert torch.isfinite(outs["1"]).all()


GROUP_HP = [(0.02, 0.01, 0.95, True), (0.05, 0.0, 0.9, False), (0.001, 0.1, 0.5, True)]


@pytest.mark.parametrize("ns_dtype", [1, 2])
def test_grouped_step_fp32_vs_oracle(capi, ns_dtype):
    """Per-group lr / wd / mu / Nesterov on the fp32 and split-fp32 paths, stage by stage
    against the oracle's grouped step (momentum and weights 1e-6, update 1e-4)."""
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    M0 = (np.random.default_rng(1).normal(0, 1e-3, M0.size)).astype(np.float32)
    group_of = [i % 3 for i in range(len(wl.shapes))]
    lay = capi.muon_layout_create(wl.shapes, 3, ns_dtype, wl.is_matrix)
    capi.muon_layout_set_groups(lay, group_of, 3)
    ws = capi.workspace_tensor(lay)
    W, M, G = split_shards(W0, 3), split_shards(M0, 3), split_shards(Gs[0], 3)
    capi.muon_step_grouped(W, G, M, lay, ws, GROUP_HP, 5)
    O = torch.zeros(lay.full_numel, device="cuda")
    capi.muon_export_update(lay, ws, 5, O)
    capi.muon_check()
    o = ref.flat_layout(wl.shapes, 1, wl.is_matrix)
    W_or, M_or, upd = ref.muon_step_grouped(W0, Gs[0], M0, o, group_of, GROUP_HP, 5)
    Wg, Mg = join_shards(W, lay.numel), join_shards(M, lay.numel)
    Og = full_to_mats(O, lay, wl)
    for i, (r, c) in enumerate(wl.shapes):
        sl = slice(o["offsets"][i], o["offsets"][i] + r * c)
        if not wl.is_matrix[i]:
            assert np.array_equal(Wg[sl], W0[sl]) and np.array_equal(Mg[sl], M0[sl])
            continue
        lr, wd, mu, nest = GROUP_HP[group_of[i]]
        assert rel(Mg[sl], M_or[sl]) < TOL_STATE, i
        parity.check_momentum(Mg[sl], M_or[sl], mu * M0[sl].astype(np.float64), i)
        parity.check_ns(Og[i], upd[i], ns_dtype, i)
        want = ref.apply_update(ref.weight_decay(W0[sl], lr, wd), Og[i].reshape(-1), lr, r, c)
        assert rel(Wg[sl], want) < TOL_STATE, i
        parity.check_weights(Wg[sl], want, W0[sl], 1 - lr * wd,
                             lr * ref.update_scale(r, c) * Og[i].reshape(-1), what=i)


def test_grouped_step_bf16_equals_ungrouped_per_group(capi):
    """On the tensor-core path each matrix's result depends only on its own group's
    values: the grouped step equals, bit for bit, the plain step run with that group's
    scalars (same layout, so the same kernels and tiles)."""
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    group_of = [i % 3 for i in range(len(wl.shapes))]
    lay = capi.muon_layout_create(wl.shapes, 2, 0, wl.is_matrix)
    capi.muon_layout_set_groups(lay, group_of, 3)
    ws = capi.workspace_tensor(lay)
    W, M, G = split_shards(W0, 2), split_shards(M0, 2), split_shards(Gs[0], 2)
    capi.muon_step_grouped(W, G, M, lay, ws, GROUP_HP, 5)
    capi.muon_check()
    Wg, Mg = join_shards(W, lay.numel), join_shards(M, lay.numel)
    o = ref.flat_layout(wl.shapes, 1, wl.is_matrix)
    for g, (lr, wd, mu, nest) in enumerate(GROUP_HP):
        W1, M1, G1 = split_shards(W0, 2), split_shards(M0, 2), split_shards(Gs[0], 2)
        capi.muon_step(W1, G1, M1, lay, ws, lr, wd, mu, nest, 5)
        capi.muon_check()
        Wu, Mu = join_shards(W1, lay.numel), join_shards(M1, lay.numel)
        for i, (r, c) in enumerate(wl.shapes):
            if wl.is_matrix[i] and group_of[i] == g:
                sl = slice(o["offsets"][i], o["offsets"][i] + r * c)
                assert np.array_equal(Wg[sl], Wu[sl]), (g, i)
                assert np.array_equal(Mg[sl], Mu[sl]), (g, i)



def test_smoke_entry_point(capi):
    """The package's smoke check (one bf16 step of the 256 x 128 case against the oracle)."""
    import __graft_entry__
    __graft_entry__.smoke()


def test_default_kernel_choice(capi, monkeypatch):
    """256 x 512 CTA-pair tiles for two Llama-3-8B layers (long reductions); CTA pairs for
    the GPT-2-small and MoE sets; single CTAs for the 32-layer set (94 TFLOP per
    iteration: long enough to run at the power limit); one launch per phase, except
    GPT-2-small (0.22 TFLOP per iteration: one persistent launch); the update applied to W
    inside the last Update on the 32-layer set only (the others run the apply pass);
    nothing on the fp32 path; an unknown pin is an error."""
    monkeypatch.delenv("MUON_TC_KERNEL", raising=False)
    monkeypatch.delenv("MUON_NS_PERSISTENT", raising=False)
    monkeypatch.delenv("MUON_FUSED_TAIL", raising=False)

    def choice(name, dtype=0):
        wl = inputs.WORKLOADS[name]
        lay = capi.muon_layout_create(wl.shapes, 1, dtype, wl.is_matrix)
        k = capi.muon_layout_ns_kernel(lay)
        k["fused"] = capi.muon_layout_fused_apply(lay)
        return k
    k = choice("llama3_8b_x2")
    assert k["tile_shape"] == 3 and not k["persistent"] and k["units"] >= 1, k
    assert not k["fused"], k
    k = choice("llama3_8b_x32")
    assert k["tile_shape"] == 1 and not k["persistent"] and k["units"] >= 1, k
    assert k["fused"], k
    k = choice("gpt2_small_x12")
    assert k["tile_shape"] == 2 and k["persistent"] and k["units"] >= 1, k
    assert not k["fused"], k
    k = choice("moe_64e")
    assert k["tile_shape"] == 2 and not k["persistent"] and k["units"] >= 1, k
    assert not k["fused"], k
    assert choice("gpt2_small_x12", 1) == {"tile_shape": 0, "units": 0, "persistent": False,
                                           "fused": False}
    monkeypatch.setenv("MUON_FUSED_TAIL", "1")
    assert choice("gpt2_small_x12")["fused"]
    monkeypatch.setenv("MUON_TC_KERNEL", "4")
    with pytest.raises(capi.MuonError) as e:
        choice("llama3_8b_x2")
    assert e.value.status == capi.MUON_ERR_INVALID_ARG


@pytest.mark.parametrize("variant", ["1", "2", "3"])
@pytest.mark.parametrize("persistent", ["0", "1"])
def test_fused_tail_each_variant(capi, variant, persistent, monkeypatch):
    """muon_step (whose last Update applies W) against the three separate stages, for each
    pinned tile shape and launch mode: momentum bit for bit, weights within the bf16
    rounding of O (2^-8 of each element, times lr * scale)."""
    monkeypatch.setenv("MUON_TC_KERNEL", variant)
    monkeypatch.setenv("MUON_NS_PERSISTENT", persistent)
    monkeypatch.setenv("MUON_FUSED_TAIL", "1")  # small sets default to the separate apply
    shapes = [(300, 200), (37, 1), (600, 1100), (520, 130), (1, 50)]
    flags = (True, False, True, True, True)
    wl = inputs.Workload("mixed_tail", tuple(shapes), flags, 2, seed=11, rank=4)
    W0, Gs, M0 = inputs.host_inputs(wl)
    res = {}
    for mode in ("step", "stages"):
        lay = capi.muon_layout_create(wl.shapes, 2, 0, wl.is_matrix)
        ws = capi.workspace_tensor(lay)
        W, M, G = split_shards(W0, 2), split_shards(M0, 2), split_shards(Gs[0], 2)
        if mode == "step":
            capi.muon_step(W, G, M, lay, ws, wl.lr, wl.wd, wl.mu, True, 5)
        else:
            capi.muon_compute_momentum_inputs(G, M, lay, ws, wl.mu, True)
            capi.muon_orthogonalize_updates(lay, ws, 5)
            capi.muon_apply_local_updates(W, lay, ws, wl.lr, wl.wd, 5)
            O = torch.zeros(lay.full_numel, device="cuda")
            capi.muon_export_update(lay, ws, 5, O)
            res["O"] = full_to_mats(O, lay, wl)
        capi.muon_check()
        res[mode] = (join_shards(W, lay.numel), join_shards(M, lay.numel))
    assert np.array_equal(res["step"][1], res["stages"][1])
    o = ref.flat_layout(wl.shapes, 1, wl.is_matrix)
    for i, Oi in res["O"].items():
        r, c = wl.shapes[i]
        sl = slice(o["offsets"][i], o["offsets"][i] + r * c)
        bound = wl.lr * ref.update_scale(r, c) * 2.0 ** -8 * (1 + 2.0 ** -8) * np.linalg.norm(Oi) \
            + 1e-6 * np.linalg.norm(res["stages"][0][sl].astype(np.float64))
        diff = np.linalg.norm(res["step"][0][sl].astype(np.float64) - res["stages"][0][sl])
        assert diff <= bound, (variant, persistent, i, diff, bound)
    v = o["offsets"][1]
    assert np.array_equal(res["step"][0][v:v + 37], W0[v:v + 37])


def test_split_fp32_matches_fp32_path_on_pair_tiles(capi):
    """The split-fp32 tensor-core path against the fp32 CUDA-core path and the oracle on
    shapes spanning several 256 x 256 pair tiles with ragged edges (tall, wide, square),
    spread spectra: both within 1e-4 of the oracle, and of each other."""
    shapes = [(600, 1100), (1100, 600), (520, 520), (257, 129), (7, 3), (64, 1000)]
    wl = inputs.Workload("tf_mixed", tuple(shapes), (True,) * len(shapes), 1, seed=12, rank=4)
    X = spectrum_inputs(wl, 21)
    got = {}
    for dt in (1, 2):
        lay = capi.muon_layout_create(wl.shapes, 1, dt, wl.is_matrix)
        if dt == 2:
            k = capi.muon_layout_ns_kernel(lay)
            assert k["tile_shape"] == 2 and not k["persistent"], k
        ws = capi.workspace_tensor(lay)
        out = torch.zeros(lay.full_numel, device="cuda")
        capi.muon_orthogonalize_full(lay, ws, mats_to_full(X, lay), out, 5)
        capi.muon_check()
        got[dt] = full_to_mats(out, lay, wl)
    for i, Xi in X.items():
        want = ref.newton_schulz(Xi.astype(np.float32).astype(np.float64), 5)
        parity.check_ns(got[2][i], want, 2, ("split", wl.shapes[i]))
        parity.check_ns(got[1][i], want, 1, ("fp32", wl.shapes[i]))
        assert rel(got[2][i], got[1][i]) < TOL_NS[2], wl.shapes[i]


@pytest.mark.parametrize("ns_dtype,variant,persistent", [(0, None, None), (0, "2", "1"),
                                                         (0, "1", "1"), (2, None, None)])
def test_step_replays_from_a_cuda_graph(capi, ns_dtype, variant, persistent, monkeypatch):
    """muon_step captured once in a CUDA graph (after a first eager call has prepared the
    layout's tables and tensor maps) and replayed for two more steps gives the same bits
    as three eager steps: per-phase launches, persistent launches of CTA pairs and of
    single CTAs, and the split-fp32 path."""
    if variant is not None:
        monkeypatch.setenv("MUON_TC_KERNEL", variant)
        monkeypatch.setenv("MUON_NS_PERSISTENT", persistent)
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    outs = []
    for mode in ("eager", "graph"):
        lay = capi.muon_layout_create(wl.shapes, 3, ns_dtype, wl.is_matrix)
        ws = capi.workspace_tensor(lay)
        W, M = split_shards(W0, 3), split_shards(M0, 3)
        G = split_shards(Gs[0], 3)
        capi.muon_step(W, G, M, lay, ws, wl.lr, wl.wd, wl.mu, True, 5)
        capi.muon_check()
        if mode == "eager":
            for _ in range(2):
                capi.muon_step(W, G, M, lay, ws, wl.lr, wl.wd, wl.mu, True, 5)
        else:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                with torch.cuda.graph(g):
                    capi.muon_step(W, G, M, lay, ws, wl.lr, wl.wd, wl.mu, True, 5)
            torch.cuda.current_stream().wait_stream(side)
            for _ in range(2):
                g.replay()
        capi.muon_check()
        outs.append((join_shards(W, lay.numel), join_shards(M, lay.numel)))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])


GUARD = 1 << 16


def guarded_workspace(lay, fill):
    """A workspace with GUARD bytes of `fill` on both sides, the workspace itself filled
    with `fill` too (1024-byte aligned)."""
    raw = torch.full((lay.workspace_bytes + 2 * GUARD + 1024,), fill, dtype=torch.uint8,
                     device="cuda")
    off = GUARD + (-(raw.data_ptr() + GUARD)) % 1024
    ws = raw[off: off + lay.workspace_bytes]
    return raw, off, ws


@pytest.mark.parametrize("ns_dtype", [0, 1, 2])
def test_workspace_guards_and_poisoned_workspace(capi, ns_dtype):
    """No kernel writes outside the workspace or reads workspace bytes it has not written:
    with the workspace and guard bands filled with 0xFF (NaN as fp32 and bf16), two steps
    give the same bits as with a zeroed workspace, and the guard bands stay 0xFF."""
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    outs = []
    for fill in (0, 0xFF):
        lay = capi.muon_layout_create(wl.shapes, 3, ns_dtype, wl.is_matrix)
        raw, off, ws = guarded_workspace(lay, fill)
        W, M = split_shards(W0, 3), split_shards(M0, 3)
        for t in range(2):
            capi.muon_step(W, split_shards(Gs[t], 3), M, lay, ws, wl.lr, wl.wd, wl.mu, True, 5)
        capi.muon_check()
        if fill == 0xFF:
            r = raw.cpu().numpy()
            assert np.all(r[:off] == 0xFF)
            assert np.all(r[off + lay.workspace_bytes:] == 0xFF)
        outs.append((join_shards(W, lay.numel), join_shards(M, lay.numel)))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("ns_dtype", [0, 2])
def test_checkpoint_resume_is_bit_exact(capi, ns_dtype):
    """Momentum is caller state: saving W and M after step 1 to the host and resuming in
    fresh buffers, a fresh layout and a fresh workspace gives step 2 bit for bit as an
    uninterrupted run."""
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    lay = capi.muon_layout_create(wl.shapes, 3, ns_dtype, wl.is_matrix)
    ws = capi.workspace_tensor(lay)
    W, M = split_shards(W0, 3), split_shards(M0, 3)
    capi.muon_step(W, split_shards(Gs[0], 3), M, lay, ws, wl.lr, wl.wd, wl.mu, True, 5)
    capi.muon_check()
    W_saved, M_saved = join_shards(W, lay.numel), join_shards(M, lay.numel)
    capi.muon_step(W, split_shards(Gs[1], 3), M, lay, ws, wl.lr, wl.wd, wl.mu, True, 5)
    capi.muon_check()
    lay2 = capi.muon_layout_create(wl.shapes, 3, ns_dtype, wl.is_matrix)
    ws2 = capi.workspace_tensor(lay2)
    W2, M2 = split_shards(W_saved, 3), split_shards(M_saved, 3)
    capi.muon_step(W2, split_shards(Gs[1], 3), M2, lay2, ws2, wl.lr, wl.wd, wl.mu, True, 5)
    capi.muon_check()
    assert np.array_equal(join_shards(W2, lay.numel), join_shards(W, lay.numel))
    assert np.array_equal(join_shards(M2, lay.numel), join_shards(M, lay.numel))

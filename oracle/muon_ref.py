"""Plain, slow fp64 CPU oracle for the sharded Muon optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links this
module; only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA path.

Sources, by page and section:

* "Add initial Muon+M-FSDPv2 implementation" (Megatron-LM pull request #6425),
  section "What does this PR do?" (every parameter placed in flat shards; one owner
  rank orthogonalizes each sharded matrix; parameters that are not matrices take the
  regular optimizer path) and its "Opt step" pseudocode, steps 1-6.
* "core.distributed.fsdp.src.megatron_fsdp.experimental.muon" (Megatron-Core API
  docs), class ``FsdpMuon``: ``_compute_momentum_inputs`` (its first stage: the
  decoupled weight decay, the momentum update and the orthogonalization input),
  ``_orthogonalize_updates`` and ``_apply_local_updates``; "Limitations" (only 2-D
  parameters take the Muon update).

The pages hand the Muon arithmetic to the base class (emerging_optimizers' Muon) and do
not print it.  This oracle takes the standard reading of that base class:

* momentum M <- mu*M + G, no dampening;
* orthogonalization input X = G + mu*M with the *updated* M (Nesterov) or X = M;
* quintic Newton-Schulz: X <- X/||X||_F, transpose so that rows <= cols, then
  ``ns_steps`` rounds of A = X X^T, B = b*A + c*A@A, X <- a*X + B@X with
  (a, b, c) = (3.4445, -4.7750, 2.0315), transposed back at the end; a zero input
  gives a zero output (no epsilon);
* decoupled weight decay W <- W*(1 - lr*wd) in the first stage (as
  ``_compute_momentum_inputs`` lists it), then W <- W - lr*sqrt(max(1, rows/cols))*O.

Flat layout (the pages place every parameter in flat shards but fix no padding): parameters
packed back to back in the given order with no padding, N elements in all; with S
shards each shard holds L = ceil(N/S) elements, shard s covering flat [s*L, (s+1)*L);
the tail of the last shard is padding and is never touched.

Every function below is pinned by tests/test_oracle.py against something other than
itself (closed form, SVD route, invariants, brute force).
"""
from __future__ import annotations

import math

import numpy as np

# Quintic Newton-Schulz coefficients of the base-class reading above.
NS_A = 3.4445
NS_B = -4.7750
NS_C = 2.0315


# --------------------------------------------------------------------------------------
# Flat layout and owner gather / scatter
# ("Add initial Muon+M-FSDPv2 implementation", "What does this PR do?" and
#  "Opt step" steps 3 and 5)
# --------------------------------------------------------------------------------------
def flat_layout(shapes, n_shards=1, is_matrix=None):
    """Describe where each parameter lives in the flat buffer and its shards.

    ``shapes`` is a list of (rows, cols); a non-matrix parameter (``is_matrix[i]`` false)
    is given as (numel, 1).  Returns a dict with per-parameter flat offsets and numels,
    the total N and the shard length L = ceil(N / n_shards).
    """
    if n_shards < 1:
        raise ValueError("n_shards must be >= 1")
    shapes = [(int(r), int(c)) for r, c in shapes]
    if is_matrix is None:
        is_matrix = [True] * len(shapes)
    is_matrix = [bool(f) for f in is_matrix]
    offsets = []
    numels = []
    pos = 0
    for (r, c) in shapes:
        offsets.append(pos)
        numels.append(r * c)
        pos += r * c
    N = pos
    L = -(-N // n_shards)  # ceil
    return {
        "shapes": shapes,
        "is_matrix": is_matrix,
        "offsets": offsets,
        "numels": numels,
        "N": N,
        "n_shards": n_shards,
        "L": L,
    }


def shard_flat(flat, layout):
    """Split an unsharded flat vector into the layout's shards (last one zero-padded)."""
    L, S, N = layout["L"], layout["n_shards"], layout["N"]
    flat = np.asarray(flat)
    shards = []
    for s in range(S):
        sh = np.zeros(L, dtype=flat.dtype)
        lo, hi = s * L, min((s + 1) * L, N)
        if hi > lo:
            sh[: hi - lo] = flat[lo:hi]
        shards.append(sh)
    return shards


def unshard_flat(shards, layout):
    """Concatenate shards back into the unsharded flat vector of length N."""
    return np.concatenate([np.asarray(s) for s in shards])[: layout["N"]]


def gather_full(shards, layout):
    """Owner gather: rebuild each matrix parameter, row-major, from its flat slices.

    Returns {param index: rows x cols array}.  A parameter's slice may straddle any
    number of shard edges; the gather is pure indexing.
    """
    flat = unshard_flat(shards, layout)
    out = {}
    for i, (r, c) in enumerate(layout["shapes"]):
        if not layout["is_matrix"][i]:
            continue
        off = layout["offsets"][i]
        out[i] = flat[off: off + r * c].reshape(r, c).copy()
    return out


def scatter_updates(full, layout, shards):
    """Owner scatter: write each full matrix back to its flat slices in the shards.

    Positions that belong to no matrix in ``full`` (non-matrix parameters, padding)
    are left unchanged.  Returns new shard arrays.
    """
    L = layout["L"]
    out = [np.array(s, copy=True) for s in shards]
    for i, mat in full.items():
        off = layout["offsets"][i]
        vals = np.asarray(mat).reshape(-1)
        for e in range(vals.size):
            g = off + e
            out[g // L][g % L] = vals[e]
    return out


# --------------------------------------------------------------------------------------
# Stage 1: weight decay, momentum, orthogonalization input
# ("Opt step" steps 1-2; FsdpMuon._compute_momentum_inputs)
# --------------------------------------------------------------------------------------
def weight_decay(W, lr, wd):
    """Decoupled weight decay: W * (1 - lr*wd)."""
    return np.asarray(W, dtype=np.float64) * (1.0 - lr * wd)


def momentum_update(M, G, mu):
    """M <- mu*M + G."""
    return mu * np.asarray(M, dtype=np.float64) + np.asarray(G, dtype=np.float64)


def ns_input(G, M_new, mu, nesterov):
    """Orthogonalization input: G + mu*M_new with Nesterov, else M_new."""
    G = np.asarray(G, dtype=np.float64)
    M_new = np.asarray(M_new, dtype=np.float64)
    return G + mu * M_new if nesterov else M_new.copy()


# --------------------------------------------------------------------------------------
# Stage 2: orthogonalization on the owner ("Opt step" step 4;
# FsdpMuon._orthogonalize_updates)
# --------------------------------------------------------------------------------------
def newton_schulz(X, ns_steps=5, coeffs=(NS_A, NS_B, NS_C)):
    """Quintic Newton-Schulz orthogonalization of one full matrix, in fp64."""
    a, b, c = coeffs
    X = np.asarray(X, dtype=np.float64)
    if X.ndim != 2:
        raise ValueError("newton_schulz wants a 2-D matrix")
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    nu = math.sqrt(float(np.sum(X * X)))
    if nu == 0.0:
        out = np.zeros_like(X)
        return out.T if transposed else out
    X = X / nu
    for _ in range(ns_steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T.copy() if transposed else X


# --------------------------------------------------------------------------------------
# Stage 3: apply the shape-scaled update ("Opt step" step 6;
# FsdpMuon._apply_local_updates)
# --------------------------------------------------------------------------------------
def update_scale(rows, cols):
    """sqrt(max(1, rows/cols)) for a stored rows x cols matrix."""
    return math.sqrt(max(1.0, rows / cols))


def apply_update(W_decayed, O, lr, rows, cols):
    """W <- W - lr * sqrt(max(1, rows/cols)) * O."""
    return np.asarray(W_decayed, dtype=np.float64) - lr * update_scale(rows, cols) * np.asarray(
        O, dtype=np.float64)


# --------------------------------------------------------------------------------------
# Whole step
# --------------------------------------------------------------------------------------
def muon_step(W, G, M, layout, lr, wd, mu, nesterov=True, ns_steps=5):
    """One unsharded optimizer step over a flat buffer (the numerics baseline).

    ``W``, ``G``, ``M`` are flat length-N vectors.  Returns (W_new, M_new, updates)
    where ``updates`` maps each matrix parameter index to its full orthogonalized
    update O.  Non-matrix parameters are skipped: their W and M bytes come back as
    they went in.
    """
    W = np.array(W, dtype=np.float64, copy=True)
    M = np.array(M, dtype=np.float64, copy=True)
    G = np.asarray(G, dtype=np.float64)
    updates = {}
    for i, (r, c) in enumerate(layout["shapes"]):
        if not layout["is_matrix"][i]:
            continue
        sl = slice(layout["offsets"][i], layout["offsets"][i] + r * c)
        Wd = weight_decay(W[sl], lr, wd)
        M[sl] = momentum_update(M[sl], G[sl], mu)
        X = ns_input(G[sl], M[sl], mu, nesterov).reshape(r, c)
        O = newton_schulz(X, ns_steps)
        updates[i] = O
        W[sl] = apply_update(Wd, O.reshape(-1), lr, r, c)
    return W, M, updates


def muon_step_sharded(W_shards, G_shards, M_shards, layout, lr, wd, mu, nesterov=True,
                      ns_steps=5):
    """The owner-based sharded step, written the way the pseudocode orders it.

    Steps 1-2 run on each shard's local slices, step 3 gathers the full inputs, step 4
    orthogonalizes, step 5 scatters the full updates back to shard order and step 6
    applies them to the local slices.  Returns (W_shards, M_shards, updates).
    """
    L = layout["L"]
    W_sh = [np.array(s, dtype=np.float64, copy=True) for s in W_shards]
    M_sh = [np.array(s, dtype=np.float64, copy=True) for s in M_shards]
    G_sh = [np.asarray(s, dtype=np.float64) for s in G_shards]
    X_sh = [np.zeros(L) for _ in range(layout["n_shards"])]
    owned = np.zeros(layout["n_shards"] * L, dtype=bool)
    for i, (r, c) in enumerate(layout["shapes"]):
        if layout["is_matrix"][i]:
            owned[layout["offsets"][i]: layout["offsets"][i] + r * c] = True
    # Steps 1-2 (and the decay) on every local shard.
    for s in range(layout["n_shards"]):
        loc = owned[s * L: (s + 1) * L]
        W_sh[s][loc] = weight_decay(W_sh[s][loc], lr, wd)
        M_sh[s][loc] = momentum_update(M_sh[s][loc], G_sh[s][loc], mu)
        X_sh[s][loc] = ns_input(G_sh[s][loc], M_sh[s][loc], mu, nesterov)
    # Step 3: gather; step 4: orthogonalize.
    full_in = gather_full(X_sh, layout)
    updates = {i: newton_schulz(X, ns_steps) for i, X in full_in.items()}
    # Step 5: scatter the scaled updates; step 6: apply locally.
    scaled = {}
    for i, O in updates.items():
        r, c = layout["shapes"][i]
        scaled[i] = lr * update_scale(r, c) * O
    U_sh = scatter_updates(scaled, layout, [np.zeros(L) for _ in range(layout["n_shards"])])
    for s in range(layout["n_shards"]):
        loc = owned[s * L: (s + 1) * L]
        W_sh[s][loc] = W_sh[s][loc] - U_sh[s][loc]
    return W_sh, M_sh, updates


def muon_step_grouped(W, G, M, layout, group_of, hparams, ns_steps=5):
    """One step with per-group hyper-parameters (Megatron-Core API page, class
    _FsdpGroupAssignment: tensor_to_optimizer_group_index maps each tensor to the
    optimizer group whose settings it uses).  ``group_of[i]`` is parameter i's group;
    ``hparams[g]`` = (lr, wd, mu, nesterov).  Returns (W_new, M_new, updates)."""
    W = np.array(W, dtype=np.float64, copy=True)
    M = np.array(M, dtype=np.float64, copy=True)
    G = np.asarray(G, dtype=np.float64)
    updates = {}
    for i, (r, c) in enumerate(layout["shapes"]):
        if not layout["is_matrix"][i]:
            continue
        lr, wd, mu, nesterov = hparams[group_of[i]]
        sl = slice(layout["offsets"][i], layout["offsets"][i] + r * c)
        Wd = weight_decay(W[sl], lr, wd)
        M[sl] = momentum_update(M[sl], G[sl], mu)
        X = ns_input(G[sl], M[sl], mu, nesterov).reshape(r, c)
        O = newton_schulz(X, ns_steps)
        updates[i] = O
        W[sl] = apply_update(Wd, O.reshape(-1), lr, r, c)
    return W, M, updates


# --------------------------------------------------------------------------------------
# Owner choice ("Add initial Muon+M-FSDPv2 implementation", "What does this PR do?": one
# owner holding at least one shard of the matrix; "Opt step" step 3: picked by
# orthogonalization compute cost).  The pages give no rule beyond that; this oracle
# reads it as longest-processing-time first onto the least-loaded eligible rank.
# --------------------------------------------------------------------------------------
def ns_cost(rows, cols, ns_steps=5):
    """Newton-Schulz flops of one matrix with symmetric Gram and A^2 (per the iteration:
    m^2 n + m^3 + 2 m^2 n per step, m = min, n = max of the shape)."""
    m, n = min(rows, cols), max(rows, cols)
    return ns_steps * (m * m * n + m ** 3 + 2 * m * m * n)


def shards_of(layout, i):
    """The shard indices holding a part of parameter i."""
    r, c = layout["shapes"][i]
    L = layout["L"]
    first = layout["offsets"][i] // L
    last = (layout["offsets"][i] + r * c - 1) // L
    return list(range(first, last + 1))


def assign_owners(layout, ns_steps=5):
    """(owner per parameter, cost per rank): each matrix, most expensive first (ties in
    parameter order), to the least-loaded rank among its shards (ties: lowest rank)."""
    S = layout["n_shards"]
    load = [0.0] * S
    owner = [-1] * len(layout["shapes"])
    jobs = [(ns_cost(r, c, ns_steps), i) for i, (r, c) in enumerate(layout["shapes"])
            if layout["is_matrix"][i]]
    jobs.sort(key=lambda t: (-t[0], t[1]))
    for cost, i in jobs:
        cands = shards_of(layout, i)
        best = min(cands, key=lambda s: (load[s], s))
        owner[i] = best
        load[best] += cost
    return owner, load

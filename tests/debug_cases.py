"""The small GPU cases run under both the release and the debug build of the library.

    MUON_LIB=.../libmuon_debug.so python -m tests.debug_cases OUT.npz

runs every case with whichever library the binding loads, checks that muon_check reports
nothing after each one (a failed range check would report MUON_ERR_DEVICE_CHECK), and
saves the results.  tests/test_gpu_debug_build.py compares them bit for bit with the
release build's.
"""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# (name, ns_dtype, pinned tile shape, pinned launch mode)
STEP_CASES = [("bf16_single", 0, "1", "0"), ("bf16_pair", 0, "2", "0"),
              ("bf16_single_persistent", 0, "1", "1"), ("bf16_pair_persistent", 0, "2", "1"),
              ("fp32", 1, None, None), ("split", 2, None, None)]


def _shards(torch, flat, n):
    L = -(-flat.size // n)
    pad = np.zeros(L * n, dtype=np.float32)
    pad[: flat.size] = flat
    return [torch.from_numpy(pad[s * L:(s + 1) * L].copy()).cuda() for s in range(n)]


def _join(shards, N):
    return np.concatenate([s.cpu().numpy() for s in shards])[:N]


def run_cases():
    import torch
    from muon_optimizer_step_gb300 import capi, inputs

    out = {}
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    saved = {k: os.environ.get(k) for k in ("MUON_TC_KERNEL", "MUON_NS_PERSISTENT")}
    try:
        for name, dt, shape, pers in STEP_CASES:
            for k, v in (("MUON_TC_KERNEL", shape), ("MUON_NS_PERSISTENT", pers)):
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
            lay = capi.muon_layout_create(wl.shapes, 3, dt, wl.is_matrix)
            ws = capi.workspace_tensor(lay)
            W, M = _shards(torch, W0, 3), _shards(torch, M0, 3)
            for t in range(2):
                capi.muon_step(W, _shards(torch, Gs[t], 3), M, lay, ws, wl.lr, wl.wd, wl.mu,
                               True, 5)
            O = torch.zeros(lay.full_numel, device="cuda")
            capi.muon_export_update(lay, ws, 5, O)
            capi.muon_check()
            out[name + "_W"] = _join(W, lay.numel)
            out[name + "_M"] = _join(M, lay.numel)
            out[name + "_O"] = O.cpu().numpy()
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    # gather / scatter over straddling shards
    lay = capi.muon_layout_create(wl.shapes, 7, 0, wl.is_matrix)
    flat = np.random.default_rng(1).normal(size=lay.numel).astype(np.float32)
    full = torch.zeros(lay.full_numel, device="cuda")
    capi.muon_gather_full(lay, _shards(torch, flat, 7), full)
    back = _shards(torch, np.zeros(lay.numel, dtype=np.float32), 7)
    capi.muon_scatter_updates(lay, full, back)
    capi.muon_check()
    out["gather"] = full.cpu().numpy()
    out["scatter"] = _join(back, lay.numel)
    # the orthogonalization of given matrices, allocating and allocation-free (fp32)
    lay = capi.muon_layout_create(wl.shapes, 1, 1, wl.is_matrix)
    ws = capi.workspace_tensor(lay)
    fin = torch.from_numpy(np.random.default_rng(2).normal(size=lay.full_numel)
                           .astype(np.float32)).cuda()
    o1 = torch.zeros(lay.full_numel, device="cuda")
    o2 = torch.zeros(lay.full_numel, device="cuda")
    capi.muon_orthogonalize_full(lay, ws, fin, o1, 5)
    capi.muon_orthogonalize_full_noalloc(lay, fin, o2, 5)
    capi.muon_check()
    out["full_fp32"] = o1.cpu().numpy()
    out["full_noalloc"] = o2.cpu().numpy()
    out["debug_build"] = np.array([1 if capi.muon_debug_build() else 0])
    return out


if __name__ == "__main__":
    np.savez(sys.argv[1], **run_cases())

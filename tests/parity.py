"""Parity checks shared by the GPU tests: whole-matrix, per-tile and per-element bounds.

A whole-matrix relative Frobenius error cannot see one wrong tile of a large matrix: on a
14336 x 4096 update a wrong 128 x 128 block moves it by about sqrt(16384 / 5.9e7) = 1.7e-2
of its norm, under the 2e-2 bound of the bf16 path.  So every Newton-Schulz output is
also checked

* per 128 x 128 block (ragged last row and column blocks included): the block's own
  relative Frobenius error stays under the same bound as the whole matrix;
* per element: |O_gpu - O_ref| <= k * 2^-8 * max|O_ref| on the bf16 path (bf16 keeps 8
  significant bits; k absorbs the rounding the iterations amplify), and
  k * tol * max|O_ref| on the fp32-accurate paths.

Momentum and weights are checked element by element:
|x_gpu - x_ref| <= 1e-6 |x_ref| + floor, with an fp32 rounding floor derived from the
arithmetic of each update (see the functions).

These helpers hold no optimizer arithmetic: they compare arrays.  The references come
from the oracle.
"""
from __future__ import annotations

import numpy as np

BLOCK = 128
BF16_REL = 2.0 ** -8          # bf16 rounding, relative to the value (8 significant bits)
FP32_REL = 2.0 ** -24         # fp32 rounding, relative (half an ulp of 24 bits)
# Per-element factor k of the Newton-Schulz bound (see module docstring).  Measured on
# GB300 over every tested workload (the ragged parity set, 256 x 128, GPT-2-small, MoE and
# sampled Llama-3-8B matrices): max |O_gpu - O_ref| / (2^-8 max|O_ref|) reached 7.1 on the
# bf16 path (a 130 x 520 matrix), 5.4 at full Llama size; max |O_gpu - O_ref| /
# (1e-4 max|O_ref|) reached 0.06 (fp32) and 0.27 (split fp32).  k leaves room above those;
# a single element off by a tenth of max|O_ref| is 25.6 on the bf16 scale.
ELEM_K = {0: 12.0, 1: 1.0, 2: 1.0}
NS_TOL = {0: 2e-2, 1: 1e-4, 2: 1e-4}
STATE_TOL = 1e-6


def rel(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    d = np.linalg.norm(y)
    return float(np.linalg.norm(x - y) / d) if d > 0 else float(np.linalg.norm(x))


def block_errors(got, want, block=BLOCK):
    """Relative Frobenius error of every block x block tile of two equal-shape matrices
    (ragged edges form smaller tiles).  A tile whose reference is zero reports its
    absolute error norm instead.  Returns a 2-D array indexed by tile row and column."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape and got.ndim == 2
    r, c = want.shape
    nr, nc = -(-r // block), -(-c // block)
    out = np.zeros((nr, nc))
    d2 = (got - want) ** 2
    w2 = want ** 2
    for bi in range(nr):
        rs = slice(bi * block, min(r, (bi + 1) * block))
        # column sums of the row band, then per tile
        dcol = d2[rs].sum(axis=0)
        wcol = w2[rs].sum(axis=0)
        for bj in range(nc):
            cs = slice(bj * block, min(c, (bj + 1) * block))
            dn = np.sqrt(dcol[cs].sum())
            wn = np.sqrt(wcol[cs].sum())
            out[bi, bj] = dn / wn if wn > 0 else dn
    return out


def ns_report(got, want, ns_dtype):
    """Whole-matrix error, worst tile error (and where), and the per-element ratio
    max|got - want| / (2^-8 max|want|) (bf16) or / (tol max|want|) (fp32 paths)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    be = block_errors(got, want)
    worst = np.unravel_index(int(np.argmax(be)), be.shape)
    scale = np.max(np.abs(want))
    unit = BF16_REL if ns_dtype == 0 else NS_TOL[ns_dtype]
    elem = float(np.max(np.abs(got - want)) / (unit * scale)) if scale > 0 else \
        float(np.max(np.abs(got)))
    return {"rel": rel(got, want), "block_max": float(be.max()), "block_at": tuple(int(v) for v in worst),
            "elem_ratio": elem}


def check_ns(got, want, ns_dtype, what=""):
    """Asserts the three Newton-Schulz bounds; returns the report."""
    rep = ns_report(got, want, ns_dtype)
    tol = NS_TOL[ns_dtype]
    assert rep["rel"] < tol, ("whole matrix", what, rep)
    assert rep["block_max"] < tol, ("128x128 block", what, rep)
    assert rep["elem_ratio"] <= ELEM_K[ns_dtype], ("element", what, rep)
    return rep


def check_momentum(got, want, mu_m_prev=0.0, what=""):
    """M <- mu*M + G is one fused multiply-add in fp32: the exact value of its fp32 inputs
    rounded once (2^-24 |M_ref|), with mu itself rounded to fp32 (2^-24 |mu*M_prev|, which
    cancellation can make large against |M_ref|).  So per element
    |M_gpu - M_ref| <= 1e-6 |M_ref| + 2^-24 (|M_ref| + |mu*M_prev|)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    bound = STATE_TOL * np.abs(want) + FP32_REL * (np.abs(want) + np.abs(mu_m_prev))
    bad = np.abs(got - want) > bound
    assert not bad.any(), ("momentum", what, int(bad.sum()), _first_bad(got, want, bad))


def check_input(got, want, g, ns_dtype, what=""):
    """The stored orthogonalization input X = G + mu*M (or M), per element: two fp32 fused
    multiply-adds (M, then X) and mu rounded to fp32 give at most 2^-20 (|X_ref| + |G|);
    the bf16 path then rounds to 8 significant bits (2^-8 |X_ref|), the split-fp32 path
    keeps h + m + l within 2^-26."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    bound = 2.0 ** -20 * (np.abs(want) + np.abs(np.asarray(g, dtype=np.float64)))
    if ns_dtype == 0:
        bound = bound + BF16_REL * np.abs(want)
    bad = np.abs(got - want) > bound
    assert not bad.any(), ("input", what, int(bad.sum()), _first_bad(got, want, bad))


def weight_floor(w_prev, decay, lrs_o):
    """fp32 rounding floor of W <- fl(W * decay) - lr*s*O (one multiply, one fused
    multiply-add, decay and lr*s themselves rounded to fp32): at most four roundings of
    2^-24 of the terms involved, so 2^-22 (|W_prev * decay| + |lr*s*O|)."""
    return 4 * FP32_REL * (np.abs(np.asarray(w_prev, dtype=np.float64) * decay) + np.abs(lrs_o))


def check_weights(got, want, w_prev, decay, lrs_o, extra=0.0, what=""):
    """|W_gpu - W_ref| <= 1e-6 |W_ref| + the fp32 rounding floor + extra (per element;
    `extra` carries a known rounding of O, e.g. lr*s*2^-8*|O| for the fused tail)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    bound = STATE_TOL * np.abs(want) + weight_floor(w_prev, decay, lrs_o) + extra
    bad = np.abs(got - want) > bound
    assert not bad.any(), ("weights", what, int(bad.sum()), _first_bad(got, want, bad))


def _first_bad(got, want, bad):
    k = int(np.flatnonzero(bad.reshape(-1))[0])
    return {"index": k, "got": float(got.reshape(-1)[k]), "want": float(want.reshape(-1)[k])}


def bf16_round(x):
    """Round fp32 values to the nearest bf16 (ties to even), returned as fp32: the upper
    16 bits of the fp32 pattern after adding 0x7FFF plus the lowest kept bit."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)

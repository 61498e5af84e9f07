"""The GPU tests' parity checks catch what a whole-matrix Frobenius bound misses.

Run on the CPU with host arrays only: an oracle output, a copy rounded to bf16 (what a
correct bf16 path stores), and that copy with one 32 x 32 block or one element planted
wrong.  The planted mistakes sit in host copies; no kernel runs.
"""
import numpy as np
import pytest

from oracle import muon_ref as ref
from tests import parity


def _ns_pair(rows, cols, seed=0):
    """(oracle output, its bf16 rounding) for a gradient-like input (noise plus rank 8)."""
    rng = np.random.default_rng(seed)
    X = rng.normal(0, 1e-3, (rows, cols)) + rng.normal(size=(rows, 8)) @ rng.normal(size=(8, cols)) * 1e-3
    O = ref.newton_schulz(X, 5)
    return O, parity.bf16_round(O).astype(np.float64)


def test_bf16_round_is_round_to_nearest_even():
    # values exactly representable, halfway cases (ties go to the even mantissa), and a
    # value just above a halfway point
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -7)
    xs = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20,
                   -1.5, 3.0e-3], dtype=np.float32)
    got = parity.bf16_round(xs)
    assert got[0] == one
    assert got[1] == one                      # tie: 1 + 2^-8 -> 1 (even)
    assert got[2] == one + 2 * ulp            # tie: 1 + 3*2^-8 -> 1 + 2^-6 (even)
    assert got[3] == one + ulp                # above the tie: up
    assert got[4] == np.float32(-1.5)
    assert abs(float(got[5]) - 3.0e-3) <= 2.0 ** -8 * 3.0e-3


def test_correct_bf16_output_passes_every_check():
    O, Ob = _ns_pair(512, 384)
    rep = parity.check_ns(Ob, O, 0, "bf16-rounded oracle")
    assert rep["elem_ratio"] <= 1.0 + 1e-9  # one bf16 rounding is within 2^-8 of max|O|


@pytest.mark.parametrize("at", [(0, 0), (13, 7), (15, 11)])  # includes the last (ragged) tile
def test_one_wrong_32x32_block_is_caught_where_frobenius_is_not(at):
    O, Ob = _ns_pair(520, 360, seed=1)
    bad = Ob.copy()
    i0, j0 = 32 * at[0], 32 * at[1]
    blk = bad[i0:i0 + 32, j0:j0 + 32]
    # a plausible-looking but wrong block: scaled so that the whole matrix moves by 1.5e-2
    # of its norm
    f = 1.5e-2 * np.linalg.norm(O) / np.linalg.norm(blk)
    bad[i0:i0 + 32, j0:j0 + 32] = (1.0 + f) * blk
    # the whole-matrix bound alone would pass it...
    assert parity.rel(bad, O) < parity.NS_TOL[0]
    # ...the per-tile check does not
    with pytest.raises(AssertionError, match="128x128 block"):
        parity.check_ns(bad, O, 0, "planted block")


def test_one_wrong_element_is_caught():
    O, Ob = _ns_pair(300, 200, seed=2)
    bad = Ob.copy()
    bad[299, 199] += 0.1 * np.max(np.abs(O))   # last row and column
    assert parity.rel(bad, O) < parity.NS_TOL[0]
    with pytest.raises(AssertionError):
        parity.check_ns(bad, O, 0, "planted element")


def test_state_checks_catch_one_element_under_a_frobenius_bound():
    rng = np.random.default_rng(3)
    G = rng.normal(0, 1e-3, 32768).astype(np.float32)
    M0 = rng.normal(0, 1e-3, 32768).astype(np.float32)
    M_ref = ref.momentum_update(M0, G, 0.95)
    # fp32 fused multiply-add, as on the GPU: the product of two fp32 values is exact in
    # fp64, the sum then rounds once more to fp32
    M_gpu = (np.float64(np.float32(0.95)) * M0 + G.astype(np.float64)).astype(np.float32)
    parity.check_momentum(M_gpu, M_ref, 0.95 * M0)
    bad = M_gpu.astype(np.float64).copy()
    bad[12345] *= 1.0 + 1e-4
    assert parity.rel(bad, M_ref) < parity.STATE_TOL
    with pytest.raises(AssertionError, match="momentum"):
        parity.check_momentum(bad, M_ref, 0.95 * M0)
    # weights: W <- W (1 - lr wd) - lr s O, in fp32 against fp64
    W0 = rng.normal(0, 0.02, 32768).astype(np.float32)
    O = rng.normal(0, 1.0 / 128, 32768).astype(np.float32)
    lr, wd, s = 0.02, 0.01, np.sqrt(2.0)
    decay = np.float32(1.0 - lr * wd)
    lrs = np.float32(lr) * np.float32(s)
    W_gpu = (W0 * decay - lrs * O).astype(np.float32)
    W_ref = ref.apply_update(ref.weight_decay(W0, lr, wd), O, lr, 256, 128)
    parity.check_weights(W_gpu, W_ref, W0, 1 - lr * wd, lr * s * O.astype(np.float64))
    badw = W_gpu.astype(np.float64).copy()
    badw[-1] += 1e-5 * abs(badw[-1]) + 1e-9
    assert parity.rel(badw, W_ref) < parity.STATE_TOL
    with pytest.raises(AssertionError, match="weights"):
        parity.check_weights(badw, W_ref, W0, 1 - lr * wd, lr * s * O.astype(np.float64))

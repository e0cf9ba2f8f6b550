"""The per-slice gradient comparison catches what a whole-tensor norm hides:
an error confined to one head, one row of one head, or one short sequence of
a packed batch; and it does not fail slices whose exact gradient is zero when
the result carries only fp32-sized residue."""
import numpy as np
import pytest

from gradcheck import check_grads, dense_slices, packed_slices


def _ref(shape, seed=0):
    return np.random.default_rng(seed).standard_normal(shape)


def _noisy(r, rel, seed=1):
    return r + rel * np.abs(r).mean() * np.random.default_rng(seed).standard_normal(r.shape)


def test_clean_result_passes():
    r = _ref((2, 8, 64, 16))
    g = _noisy(r, 2e-3)
    check_grads([g] * 3, [r] * 3, dense_slices(2, 8))


def test_one_bad_head_fails_although_the_global_norm_passes():
    B, H = 2, 128
    r = _ref((B, H, 32, 16))
    g = r.copy()
    g[1, 77] *= 1.10  # 10 % off on one head of 256
    glob = np.linalg.norm(g - r) / np.linalg.norm(r)
    assert glob < 1e-2  # a whole-tensor norm would accept it
    with pytest.raises(AssertionError, match=r"\(1, 77\)"):
        check_grads([g, r, r], [r, r, r], dense_slices(B, H))


def test_one_wrong_row_fails_the_elementwise_bound():
    r = _ref((1, 2, 512, 64))
    g = r.copy()
    g[0, 1, 300, :2] += 0.05 * np.abs(r[0, 1]).max()  # two elements of one row
    assert np.linalg.norm(g[0, 1] - r[0, 1]) / np.linalg.norm(r[0, 1]) < 1e-2
    with pytest.raises(AssertionError, match="dK"):
        check_grads([r, g, r], [r, r, r], dense_slices(1, 2))


def test_zero_reference_slice_accepts_fp32_residue_only():
    r = _ref((1, 3, 16, 8))
    r[0, 2] = 0.0  # e.g. a head that sees a single key: dQ = dK = 0 exactly
    g = r.copy()
    g[0, 2] = 1e-7 * _ref((16, 8), 5)
    check_grads([g] * 3, [r] * 3, dense_slices(1, 3))
    g[0, 2] = 0.1 * _ref((16, 8), 5)  # but not a real error
    with pytest.raises(AssertionError):
        check_grads([g] * 3, [r] * 3, dense_slices(1, 3))


def test_packed_short_sequence_is_judged_on_its_own():
    lens = [1000, 17, 1000]
    cu = np.concatenate([[0], np.cumsum(lens)])
    H = 2
    r = _ref((int(cu[-1]), H, 32))
    g = r.copy()
    g[cu[1]:cu[2], 1] *= 1.1  # the 17-token sequence, one head
    assert np.linalg.norm(g - r) / np.linalg.norm(r) < 1e-2
    with pytest.raises(AssertionError, match=r"\(1, 1\)"):
        check_grads([g, r, r], [r, r, r], packed_slices(cu, H))
    check_grads([r, r, r], [r, r, r], packed_slices(cu, H))


def test_whole_tensor_zero_uses_the_other_gradients_scale():
    # one key per row: dQ = dK = 0 everywhere, dV = dO
    dv = _ref((2, 2, 1, 64))
    z = np.zeros_like(dv)
    res = 1e-7 * _ref(dv.shape, 9)
    check_grads([res, res, dv], [z, z, dv], dense_slices(2, 2))
    with pytest.raises(AssertionError, match="dQ"):
        check_grads([1e-2 * _ref(dv.shape, 9), res, dv], [z, z, dv], dense_slices(2, 2))

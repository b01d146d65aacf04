"""Host checks of the seeded input generators (no GPU): the recipe that the
tests and the bench feed to both the library and the oracle."""

import numpy as np
import torch

from rotated_int2_kv_gb300 import synth

SEED = 1234


def test_tokens_are_a_function_of_position():
    # any chunking of the appends sees the same values: rows p0 .. p0+n-1 drawn
    # alone equal the same rows of a longer draw, across a block boundary
    scales = synth.outlier_scales(SEED, 2, 64, "fixed4")
    k_all, v_all = synth.kv_tokens(SEED, 3, 0, 3 * synth.BLOCK, 2, 64, scales)
    for p0, n in ((0, 1), (1000, 100), (synth.BLOCK - 1, 2), (2 * synth.BLOCK + 5, 7)):
        k, v = synth.kv_tokens(SEED, 3, p0, n, 2, 64, scales)
        assert torch.equal(k, k_all[p0:p0 + n]) and torch.equal(v, v_all[p0:p0 + n])
    # other requests and other seeds draw other values
    k_other, _ = synth.kv_tokens(SEED, 4, 0, 16, 2, 64, scales)
    assert not torch.equal(k_other, k_all[:16])
    k_seed, _ = synth.kv_tokens(SEED + 1, 3, 0, 16, 2, 64, scales)
    assert not torch.equal(k_seed, k_all[:16])
    # an empty draw
    k0, v0 = synth.kv_tokens(SEED, 3, 10, 0, 2, 64, scales)
    assert k0.shape == (0, 2, 64) and v0.shape == (0, 2, 64)


def test_outlier_channels():
    ks, vs = synth.outlier_scales(SEED, 8, 128, "fixed4")
    ks, vs = ks.numpy(), vs.numpy()
    # four channels, the same in every KV head: x20 in K, x4 in V
    assert ((ks == 20.0).sum(axis=1) == 4).all() and ((vs == 4.0).sum(axis=1) == 4).all()
    assert (ks[:, ks[0] == 20.0] == 20.0).all()
    assert set(np.unique(ks)) == {1.0, 20.0} and set(np.unique(vs)) == {1.0, 4.0}
    kp, vp = synth.outlier_scales(SEED, 8, 128, "per_head")
    kp, vp = kp.numpy(), vp.numpy()
    n_out = (kp != 1.0).sum(axis=1)
    assert ((n_out >= 2) & (n_out <= 8)).all()
    big = kp[kp != 1.0]
    assert ((big >= 10.0) & (big <= 30.0)).all()
    assert np.array_equal(vp, vs)                       # V keeps the fixed four channels


def test_calibration_spectrum():
    # x = z diag(sqrt(lambda)) Q^T with lambda_i ~ i^-1.5: the sample covariance
    # has eigenvalues close to lambda (65,536 rows, d 32: within sampling error)
    d = 32
    X = synth.calib_samples(SEED, 0, d, n=65536)
    w = np.sort(np.linalg.eigvalsh(X.T @ X / X.shape[0]))[::-1]
    lam = np.arange(1, d + 1, dtype=np.float64) ** -1.5
    assert np.abs(w / lam - 1.0).max() < 0.1
    # the key side and the value side use different orthogonal bases
    Y = synth.calib_samples(SEED, 1, d, n=65536)
    Ck, Cv = X.T @ X / X.shape[0], Y.T @ Y / Y.shape[0]
    assert np.abs(Ck - Cv).max() > 0.1


def test_page_tables_and_lengths():
    pt = synth.page_table(SEED, 4, 100, 1000).numpy()
    assert pt.shape == (4, 100) and len(np.unique(pt)) == 400
    assert pt.min() >= 0 and pt.max() < 1000
    assert not np.array_equal(pt.ravel(), np.arange(400))          # shuffled
    assert np.array_equal(synth.page_table(SEED, 4, 100, 1000, shuffled=False).numpy().ravel(), np.arange(400))
    lens = synth.ragged_lengths(SEED, 64, 65536, 131072)
    assert ((lens >= 65536) & (lens <= 131072)).all() and len(np.unique(lens)) > 32

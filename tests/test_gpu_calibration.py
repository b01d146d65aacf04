"""GPU parity of the calibration statistics (oscar_covariance_device,
oscar_value_covariance_device) against the oracle's fp64 C_Q and C_S
([OSCAR news] "OSCARの違い"), and of the rotation built from them."""

import numpy as np
import pytest
import torch

import oracle
from rotated_int2_kv_gb300 import synth

pytestmark = pytest.mark.gpu

SEED = 1234


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


@pytest.mark.parametrize("n,d", [(4096, 128), (1000, 64), (777, 256), (33, 100), (1, 8)])
def test_query_covariance_matches_oracle(n, d):
    from rotated_int2_kv_gb300 import ops
    rng = np.random.default_rng(SEED + n + d)
    X = (rng.standard_normal((n, d)) * np.where(rng.random(d) < 0.05, 20.0, 1.0)).astype(np.float32)
    got = ops.covariance_device(torch.from_numpy(X).cuda()).cpu().numpy()
    want = oracle.covariance(X.astype(np.float64))
    assert _rel(got, want) <= 1e-12
    assert np.array_equal(got, got.T)


def test_query_covariance_bf16_rows_and_determinism():
    from rotated_int2_kv_gb300 import ops
    d = 128
    X = torch.from_numpy(synth.calib_samples(SEED, 0, d).astype(np.float32)).to(torch.bfloat16)
    got = ops.covariance_device(X.cuda()).cpu().numpy()
    again = ops.covariance_device(X.cuda()).cpu().numpy()
    assert np.array_equal(got, again)                 # a fixed summation order
    want = oracle.covariance(X.float().numpy().astype(np.float64))
    assert _rel(got, want) <= 1e-12


@pytest.mark.parametrize("n_q,n_k,d,vdt", [(512, 700, 128, torch.float32), (100, 3000, 64, torch.bfloat16),
                                           (65, 33, 256, torch.float32)])
def test_value_covariance_matches_oracle(n_q, n_k, d, vdt):
    from rotated_int2_kv_gb300 import ops
    rng = np.random.default_rng(SEED + n_q)
    logits = rng.standard_normal((n_q, n_k)) * 3.0
    S = np.exp(logits - logits.max(axis=1, keepdims=True))
    S = (S / S.sum(axis=1, keepdims=True)).astype(np.float32)
    V = torch.from_numpy(rng.standard_normal((n_k, d)).astype(np.float32)).to(vdt)
    got = ops.value_covariance_device(torch.from_numpy(S).cuda(), V.cuda()).cpu().numpy()
    want = oracle.value_covariance(S.astype(np.float64), V.float().numpy().astype(np.float64))
    assert _rel(got, want) <= 1e-12


@pytest.mark.parametrize("n_q,n_k,d", [(40000, 40, 256), (64, 4000, 128)])
def test_value_covariance_split_paths_and_determinism(n_q, n_k, d):
    # (40000, 40, 256): Y fills the GPU and its partial sums would pass 64 MB, so the
    # keys are not split; (64, 4000, 128): two tiles of Y, the keys split into many
    # ranges whose partial Y are added in a fixed order
    from rotated_int2_kv_gb300 import ops
    rng = np.random.default_rng(SEED + n_k)
    S = rng.random((n_q, n_k)).astype(np.float32)
    S /= S.sum(axis=1, keepdims=True)
    V = torch.from_numpy(rng.standard_normal((n_k, d)).astype(np.float32)).to(torch.bfloat16)
    Sd, Vd = torch.from_numpy(S).cuda(), V.cuda()
    got = ops.value_covariance_device(Sd, Vd).cpu().numpy()
    again = ops.value_covariance_device(Sd, Vd).cpu().numpy()
    assert np.array_equal(got, again)
    want = oracle.value_covariance(S.astype(np.float64), V.float().numpy().astype(np.float64))
    assert _rel(got, want) <= 1e-12


def test_rotation_from_device_covariance():
    # the library's rotation from the device C_Q equals the oracle's rotation from its C_Q
    from rotated_int2_kv_gb300 import ops
    d = 128
    X = synth.calib_samples(SEED, 0, d).astype(np.float32)
    C = ops.covariance_device(torch.from_numpy(X).cuda()).cpu().numpy()
    R32, R64, w = ops.build_rotation(C, d)
    Ro, wo = oracle.build_rotation(oracle.covariance(X.astype(np.float64)), d)
    assert np.abs(w - wo).max() <= 1e-12 * np.abs(wo).max()
    assert np.abs(R64 - Ro).max() <= 1e-9

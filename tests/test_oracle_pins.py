"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: a closed
form, a brute-force definition written out independently here, a library
routine, or a figure printed on the pages (tests/golden/).
"""

import itertools
import math
import os

import numpy as np
import pytest

import oracle
from oracle import quant as oq

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# --------------------------------------------------------------------------
# rotation
# --------------------------------------------------------------------------

def test_hadamard_matches_golden_and_closed_form():
    H8 = np.array([[float(t) for t in r.split()] for r in _read_rows("sylvester_hadamard_8.txt")])
    assert np.array_equal(oracle.hadamard(8), H8)
    for n in (1, 2, 4, 16, 64, 256):
        H = oracle.hadamard(n)
        closed = np.array([[(-1.0) ** bin(i & j).count("1") for j in range(n)] for i in range(n)])
        assert np.array_equal(H, closed)
        assert np.array_equal(H @ H.T, n * np.eye(n))


def test_hadamard_256_exactly_orthogonal_in_fp32():
    # deployment log, part 2, fix 3: (rot @ rot.T - I).abs().max() == 0 for
    # the fp32 Hadamard / sqrt(256); 1/16 is dyadic so fp32 is exact.
    torch = pytest.importorskip("torch")
    rot = torch.from_numpy(oracle.hadamard(256) / math.sqrt(256)).to(torch.float32)
    assert (rot @ rot.T - torch.eye(256)).abs().max().item() == 0.0


def test_bitrev_golden_and_involution():
    br8 = [int(t) for t in _read_rows("bitrev_8.txt")[0].split()]
    assert list(oracle.bitrev_indices(8)) == br8
    for d in (2, 64, 128, 256):
        br = oracle.bitrev_indices(d)
        assert sorted(br) == list(range(d))
        assert np.array_equal(br[br], np.arange(d))
        assert br[1] == d // 2


def test_eig_desc_two_by_two_closed_form():
    rng = np.random.default_rng(1)
    for _ in range(20):
        a, c = rng.uniform(0.1, 3.0, 2)
        b = rng.uniform(-1.0, 1.0)
        w, U = oracle.eig_desc(np.array([[a, b], [b, c]]))
        mid = (a + c) / 2
        rad = math.sqrt(((a - c) / 2) ** 2 + b * b)
        assert abs(w[0] - (mid + rad)) < 1e-13 and abs(w[1] - (mid - rad)) < 1e-13
        # eigenvector of the larger eigenvalue is ∝ (b, λ1 - a)
        v = np.array([b, mid + rad - a])
        v /= np.linalg.norm(v)
        if v[np.argmax(np.abs(v))] < 0:
            v = -v
        assert np.allclose(U[:, 0], v, atol=1e-12)


def test_eig_desc_diagonal_is_sorting_permutation_and_signs():
    diag = np.array([0.3, 5.0, 1.0, 2.0])
    w, U = oracle.eig_desc(np.diag(diag))
    assert np.array_equal(w, np.array([5.0, 2.0, 1.0, 0.3]))
    expect = np.zeros((4, 4))
    for col, row in enumerate([1, 3, 2, 0]):
        expect[row, col] = 1.0
    assert np.array_equal(U, expect)


def test_eig_desc_reconstructs_random_covariance():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((512, 64)) * (np.arange(1, 65) ** -0.75)
    C = X.T @ X / 512
    w, U = oracle.eig_desc(C)
    assert np.all(np.diff(w) <= 0)
    assert np.abs(U @ np.diag(w) @ U.T - C).max() <= 1e-12 * np.abs(C).max()
    assert np.abs(U.T @ U - np.eye(64)).max() <= 1e-12
    for j in range(64):
        i = np.argmax(np.abs(U[:, j]))
        assert U[i, j] > 0


def test_rotation_without_covariance_is_the_pages_hadamard():
    # deployment log, part 2, fix 3: calibration-free rotation = Hadamard/sqrt(d)
    for d in (64, 128, 256):
        R, w = oracle.build_rotation(None, d, use_bitrev=False)
        assert w is None
        assert np.array_equal(R, oracle.hadamard(d) / math.sqrt(d))
        Rb, _ = oracle.build_rotation(None, d, use_bitrev=True)
        br = oracle.bitrev_indices(d)
        for j in (0, 1, d - 1):
            assert np.array_equal(Rb[:, j], R[:, br[j]])


def test_rotation_is_orthogonal_and_factorises():
    rng = np.random.default_rng(3)
    d = 128
    X = rng.standard_normal((4096, d)) * (np.arange(1, d + 1) ** -0.75)
    C = oracle.covariance(X)
    R, w = oracle.build_rotation(C, d)
    assert np.abs(R @ R.T - np.eye(d)).max() <= 1e-12
    # R = U · H/sqrt(d) · P  =>  R P^T H^T sqrt(d)/d = U, an eigenbasis of C
    br = oracle.bitrev_indices(d)
    P = np.zeros((d, d))
    P[br, np.arange(d)] = 1.0           # (x P)[j] = x[br[j]]
    U = R @ P.T @ oracle.hadamard(d).T / math.sqrt(d)
    assert np.abs(C @ U - U * w).max() <= 1e-10 * np.abs(C).max()


def test_block_hadamard_closed_form_and_orthogonality():
    for d, B in ((128, 16), (64, 64), (256, 32), (8, 2), (8, 1)):
        M = oracle.block_hadamard(d, B)
        assert np.abs(M @ M.T - np.eye(d)).max() <= 1e-15
        i, j = np.meshgrid(np.arange(d), np.arange(d), indexing="ij")
        same = (i // B) == (j // B)
        sign = np.array([[(-1.0) ** bin(a & b & (B - 1)).count("1") for b in range(d)] for a in range(d)])
        assert np.array_equal(M, np.where(same, sign / math.sqrt(B), 0.0))
    # the full size is the page's Hadamard
    assert np.array_equal(oracle.block_hadamard(64, 64), oracle.hadamard(64) / 8.0)
    R_full, _ = oracle.build_rotation(None, 128, hadamard_block=128)
    R_def, _ = oracle.build_rotation(None, 128)
    assert np.array_equal(R_full, R_def)


def test_bitrev_spreads_every_importance_block_over_every_group():
    # C = diag(lambda) descending: U = I, so input channel k is importance level
    # k, and block b of H_B mixes levels [bB, (b+1)B).  After P_br, every group of
    # G consecutive output channels takes G·B/d channels of every block; without
    # P_br each group sees only G/B blocks.
    d = 128
    C = np.diag(np.arange(d, 0, -1, dtype=np.float64))
    for B, G in ((16, 64), (8, 32), (32, 128), (128, 64)):
        R, _ = oracle.build_rotation(C, d, hadamard_block=B)
        for g in range(d // G):
            cols = R[:, g * G:(g + 1) * G]
            # output channels of the group fed by block b
            per_block = np.array([(np.abs(cols[b * B:(b + 1) * B]).sum(axis=0) > 0).sum()
                                  for b in range(d // B)])
            assert (per_block == G * B // d).all(), (B, G, g, per_block)
        if B < G:
            Rn, _ = oracle.build_rotation(C, d, use_bitrev=False, hadamard_block=B)
            cols = Rn[:, :G]
            per_block = np.array([(np.abs(cols[b * B:(b + 1) * B]).sum(axis=0) > 0).sum() for b in range(d // B)])
            assert (per_block[: G // B] == B).all() and (per_block[G // B:] == 0).all()


def test_covariances_against_explicit_sums():
    rng = np.random.default_rng(4)
    X = rng.standard_normal((7, 5))
    C = np.zeros((5, 5))
    for n in range(7):
        for i in range(5):
            for j in range(5):
                C[i, j] += X[n, i] * X[n, j]
    assert np.allclose(oracle.covariance(X), C / 7, rtol=0, atol=1e-14)
    S = rng.uniform(size=(3, 7))
    V = rng.standard_normal((7, 5))
    CS = np.zeros((5, 5))
    for a in range(3):
        sv = [sum(S[a, t] * V[t, i] for t in range(7)) for i in range(5)]
        for i in range(5):
            for j in range(5):
                CS[i, j] += sv[i] * sv[j]
    assert np.allclose(oracle.value_covariance(S, V), CS / 3, rtol=0, atol=1e-13)


def test_rotation_invariance_of_logits_and_attention():
    rng = np.random.default_rng(5)
    d = 128
    R, _ = oracle.build_rotation(oracle.covariance(rng.standard_normal((256, d))), d)
    q = rng.standard_normal((4, d))
    K = rng.standard_normal((50, d))
    V = rng.standard_normal((50, d))
    assert np.abs((q @ R) @ (K @ R).T - q @ K.T).max() <= 1e-12 * np.abs(q @ K.T).max()

    def attn(q, K, V):
        l = q @ K.T / math.sqrt(d)
        p = np.exp(l - l.max(axis=1, keepdims=True))
        return (p / p.sum(axis=1, keepdims=True)) @ V

    rot = attn(q @ R, K @ R, V @ R) @ R.T
    assert np.abs(rot - attn(q, K, V)).max() <= 1e-12


def test_logit_error_identity():
    # OSCAR news, "OSCARの違い": ||QKᵀ - QK̂ᵀ||_F² = tr((K-K̂) QᵀQ (K-K̂)ᵀ)
    rng = np.random.default_rng(6)
    d, G = 128, 64
    Q = rng.standard_normal((40, d))
    K = rng.standard_normal((30, d)).astype(np.float32)
    codes, s, z = oracle.quantize_rows(K, G, 0.9)
    Kh = oracle.dequantize_rows(codes, s, z)
    lhs = np.linalg.norm(Q @ K.astype(np.float64).T - Q @ Kh.T) ** 2
    E = K.astype(np.float64) - Kh
    rhs = np.trace(E @ Q.T @ Q @ E.T)
    assert abs(lhs - rhs) <= 1e-10 * abs(lhs)


# --------------------------------------------------------------------------
# quantiser and packing
# --------------------------------------------------------------------------

def test_bf16_round_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(100000) * 10 ** rng.uniform(-6, 4, 100000)).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]   # ties to even
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(oracle.bf16_round(x), ref)
    # the stored windows hold the bf16 bit patterns: torch's, and back to the values
    tb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oq.bf16_bits(ref), tb)
    assert np.array_equal(oq.bf16_from_bits(tb), ref)


def test_e4m3_rounding_matches_torch():
    # every finite E4M3 value decodes as torch's float8_e4m3fn and encodes back
    torch = pytest.importorskip("torch")
    b = np.array([i for i in range(256) if (i & 0x7F) != 0x7F], np.uint8)
    v = oq.e4m3_from_bits(b)
    assert np.array_equal(v, torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float32).numpy())
    assert np.array_equal(oq.e4m3_bits(v), b)
    assert float(v.max()) == 448.0 and float(v[v > 0].min()) == 2.0 ** -9
    # rounding to nearest, ties to even, over the range where torch's cast is finite
    rng = np.random.default_rng(70)
    x = (rng.standard_normal(200000) * 10 ** rng.uniform(-5, 2.7, 200000)).astype(np.float32)
    vs = np.unique(np.abs(v)).astype(np.float64)
    mids = ((vs[:-1] + vs[1:]) / 2).astype(np.float32)     # exact midpoints (ties)
    x = np.concatenate([x, mids, -mids])
    x = x[np.abs(x) < 464]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert np.array_equal(oracle.e4m3_round(x), ref)
    # reading: finite values beyond the largest finite one saturate (torch gives NaN)
    assert np.array_equal(oracle.e4m3_round(np.array([464, 1e6, -500], np.float32)), [448, 448, -448])
    # signed zeros survive
    z = oracle.e4m3_round(np.array([-0.0, -1e-4], np.float32))
    assert np.all(z == 0) and np.all(np.signbit(z))


def test_quantiser_exact_grid_round_trip():
    # values already on the INT2 grid come back exactly at clip ratio 1.0
    rng = np.random.default_rng(8)
    d, G = 128, 64
    n = 200
    codes = rng.integers(0, 4, size=(n, d)).astype(np.uint8)
    codes.reshape(n, d // G, G)[:, :, 0] = 0      # every group spans the full grid
    codes.reshape(n, d // G, G)[:, :, 1] = 3
    s = 2.0 ** rng.integers(-6, 3, size=(n, d // G))
    z = rng.integers(-64, 64, size=(n, d // G)) * 2.0 ** -4
    Y = (z[:, :, None] + codes.reshape(n, d // G, G) * s[:, :, None]).reshape(n, d)
    c2, s2, z2 = oracle.quantize_rows(Y.astype(np.float32), G, 1.0)
    assert np.array_equal(c2, codes)
    assert np.array_equal(s2.astype(np.float64), s)
    assert np.array_equal(z2.astype(np.float64), z)
    assert np.array_equal(oracle.dequantize_rows(c2, s2, z2), Y)


def test_quantiser_e4m3_exact_grid_round_trip():
    # with E4M3-exact s and z, values on the INT2 grid come back exactly at clip 1.0
    rng = np.random.default_rng(71)
    d, G = 128, 64
    n = 200
    codes = rng.integers(0, 4, size=(n, d)).astype(np.uint8)
    codes.reshape(n, d // G, G)[:, :, 0] = 0
    codes.reshape(n, d // G, G)[:, :, 1] = 3
    s = (1.0 + rng.integers(0, 8, size=(n, d // G)) / 8.0) * 2.0 ** rng.integers(-5, 3, size=(n, d // G))
    z = -(1.0 + rng.integers(0, 8, size=(n, d // G)) / 8.0) * 2.0 ** rng.integers(-3, 3, size=(n, d // G))
    Y = (z[:, :, None] + codes.reshape(n, d // G, G) * s[:, :, None]).reshape(n, d)
    assert np.array_equal(Y.astype(np.float32).astype(np.float64), Y)     # fp32-exact inputs
    c2, s2, z2 = oracle.quantize_rows(Y.astype(np.float32), G, 1.0, "e4m3")
    assert np.array_equal(c2, codes)
    assert np.array_equal(s2.astype(np.float64), s)
    assert np.array_equal(z2.astype(np.float64), z)
    # the f16 path would keep (hi - lo)/3 at 11 bits: scales that are not E4M3
    # values are rounded by the E4M3 path
    Y3 = np.zeros((1, 64), np.float32)
    Y3[0, 1] = 3 * 1.0625      # s = 1.0625 (fp16-exact, between E4M3 1.0 and 1.125)
    c3, s3, z3 = oracle.quantize_rows(Y3, 64, 1.0, "e4m3")
    assert float(s3[0, 0]) == 1.0 and float(z3[0, 0]) == 0.0
    c4, s4, _ = oracle.quantize_rows(Y3, 64, 1.0, "f16")
    assert float(s4[0, 0]) == 1.0625


def test_quantiser_e4m3_code_is_the_nearest_level_brute_force():
    rng = np.random.default_rng(72)
    d, G = 64, 32
    Y = (rng.standard_normal((300, d)) * 3).astype(np.float32)
    codes, s, z = oracle.quantize_rows(Y, G, 0.9, "e4m3")
    assert np.array_equal(oracle.e4m3_round(s.astype(np.float32)), s.astype(np.float32))
    assert np.array_equal(oracle.e4m3_round(z.astype(np.float32)), z.astype(np.float32))
    for i in range(300):
        for gi in range(d // G):
            yg = Y[i, gi * G:(gi + 1) * G]
            lo = np.float32(np.float32(0.9) * yg.min())
            hi = np.float32(np.float32(0.9) * yg.max())
            assert float(s[i, gi]) == float(oracle.e4m3_round(np.float32(np.float32(hi - lo) / np.float32(3))))
            assert float(z[i, gi]) == float(oracle.e4m3_round(lo))
            s32 = np.float32(s[i, gi])
            z32 = np.float32(z[i, gi])
            for j in range(gi * G, (gi + 1) * G):
                u = float(np.float32(np.float32(Y[i, j] - z32) / s32))
                best = min(range(4), key=lambda k: (abs(u - k), k))
                frac = u - math.floor(u)
                if abs(frac - 0.5) > 1e-9 or u < 0 or u > 3:
                    assert codes[i, j] == best


def test_quantiser_code_is_the_nearest_level_brute_force():
    rng = np.random.default_rng(9)
    d, G = 64, 32
    Y = (rng.standard_normal((300, d)) * 3).astype(np.float32)
    codes, s, z = oracle.quantize_rows(Y, G, 0.9)
    assert s.dtype == np.float16 and z.dtype == np.float16
    for i in range(300):
        for gi in range(d // G):
            # the stored pair is the fp16 rounding (numpy's IEEE conversion) of the
            # fp32 (hi - lo)/3 and lo of the clipped group
            yg = Y[i, gi * G:(gi + 1) * G]
            lo = np.float32(np.float32(0.9) * yg.min())
            hi = np.float32(np.float32(0.9) * yg.max())
            assert float(s[i, gi]) == float(np.float16(np.float32(np.float32(hi - lo) / np.float32(3))))
            assert float(z[i, gi]) == float(np.float16(lo))
            s32 = np.float32(s[i, gi])
            z32 = np.float32(z[i, gi])
            for j in range(gi * G, (gi + 1) * G):
                u = float(np.float32(np.float32(Y[i, j] - z32) / s32))
                best = min(range(4), key=lambda k: (abs(u - k), k))
                frac = u - math.floor(u)
                if abs(frac - 0.5) > 1e-9 or u < 0 or u > 3:
                    assert codes[i, j] == best
    # clipping: the group extreme beyond r*max saturates at code 3 (and 0 below)
    Y2 = np.zeros((1, 32), np.float32)
    Y2[0, :16] = np.linspace(-1, 1, 16)
    Y2[0, 16] = 10.0
    Y2[0, 17] = -10.0
    c, s, z = oracle.quantize_rows(Y2, 32, 0.9)
    assert c[0, 16] == 3 and c[0, 17] == 0
    assert float(z[0, 0]) == float(np.float16(np.float32(0.9) * np.float32(-10.0)))


def test_quantiser_ties_round_to_even():
    # the code of a quotient exactly halfway between two levels is the even one
    # (rint, half to even): with s = 1 and z = 0, u = 0.5, 1.5, 2.5 give 0, 2, 2
    Y = np.zeros((1, 32), np.float32)
    Y[0, 1] = 3.0                               # min 0 and max 3 at clip 1.0
    Y[0, 2:5] = [0.5, 1.5, 2.5]
    c, s, z = oracle.quantize_rows(Y, 32, 1.0)
    assert float(s[0, 0]) == 1.0 and float(z[0, 0]) == 0.0
    assert list(c[0, :5]) == [0, 3, 0, 2, 2]


def test_quantiser_flat_group():
    Y = np.full((2, 64), 1.25, np.float32)
    c, s, z = oracle.quantize_rows(Y, 64, 0.9)
    assert np.all(c == 0) and np.all(s == 0)
    assert np.all(oracle.dequantize_rows(c, s, z) == float(np.float16(np.float32(0.9) * np.float32(1.25))))


def test_packing_golden_and_round_trip():
    for line in _read_rows("pack_example.txt"):
        lhs, rhs = line.split("->")
        codes = np.array([int(t) for t in lhs.split()], np.uint8)
        expect = np.array([int(t, 16) for t in rhs.split()], np.uint8)
        assert np.array_equal(oracle.pack_codes(codes), expect)
    rng = np.random.default_rng(10)
    c = rng.integers(0, 4, (5, 3, 128)).astype(np.uint8)
    assert np.array_equal(oracle.unpack_codes(oracle.pack_codes(c)), c)


def test_record_round_trip_and_size():
    rng = np.random.default_rng(11)
    for d, G, size in ((128, 64, 80), (256, 128, 144), (128, 32, 96), (64, 64, 48)):
        ng = d // G
        kc = rng.integers(0, 4, (3, d)).astype(np.uint8)
        vc = rng.integers(0, 4, (3, d)).astype(np.uint8)
        ks, kz, vs, vz = (rng.standard_normal((3, ng)).astype(np.float16) for _ in range(4))
        rec = oq.pack_record(kc, ks, kz, vc, vs, vz, d, G)
        assert rec.shape == (3, size) and oracle.record_bytes(d, G) == size
        back = oq.unpack_record(rec, d, G)
        for a, b in zip(back, (kc, ks, kz, vc, vs, vz)):
            assert np.array_equal(a, b)


def test_e4m3_record_and_slot_layout():
    rng = np.random.default_rng(73)
    # (d, G, KV heads, record bytes, slot bytes): codes d/2 + 2-byte (s, z) pairs,
    # records padded to 8 bytes and packed back to back, slots padded to 16
    for d, G, H, rec_size, slot_size in ((128, 64, 8, 72, 576), (256, 128, 4, 136, 544),
                                         (128, 128, 3, 72, 224), (64, 64, 1, 40, 48),
                                         (128, 32, 2, 80, 160)):
        ng = d // G
        kc = rng.integers(0, 4, (5, H, d)).astype(np.uint8)
        vc = rng.integers(0, 4, (5, H, d)).astype(np.uint8)
        ks, kz, vs, vz = (oracle.e4m3_round(rng.standard_normal((5, H, ng)) * 4).astype(np.float16)
                          for _ in range(4))
        rec = oq.pack_record(kc, ks, kz, vc, vs, vz, d, G, "e4m3")
        assert rec.shape == (5, H, rec_size) and oracle.record_bytes(d, G, scale_bits=8) == rec_size
        # byte d/2 + 2gi holds the E4M3 bits of K's s of group gi, the next byte z
        assert np.array_equal(rec[..., d // 2 + 1], oq.e4m3_bits(kz[..., 0]))
        assert np.array_equal(rec[..., d // 2 + 2 * ng], oq.e4m3_bits(vs[..., 0]))
        assert oq.slot_bytes(d, G, H, "e4m3") == slot_size
        sl = oq.pack_slots(rec, slot_size)
        assert sl.shape == (5, slot_size) and not sl[:, H * rec_size:].any()
        assert np.array_equal(sl[:, rec_size:2 * rec_size] if H > 1 else sl[:, :rec_size], rec[:, min(1, H - 1)])
        assert np.array_equal(oq.head_records(sl, H, rec_size), rec)
        back = oq.unpack_record(rec, d, G, "e4m3")
        for a, b in zip(back, (kc, ks, kz, vc, vs, vz)):
            assert np.array_equal(a, b)
    # the fp16 slot is the per-head records back to back (records already 16-byte multiples)
    assert oq.slot_bytes(128, 64, 8) == 640


# --------------------------------------------------------------------------
# accounting (figures printed on the pages)
# --------------------------------------------------------------------------

def test_accounting_matches_pages():
    gold = {}
    for line in _read_rows("accounting.txt"):
        k, v = line.split()
        gold[k] = float(v)
    assert oracle.code_bytes_per_token(16, 4, 256) / 1024 == gold["kib_per_token_16x4_d256"]
    assert oracle.code_bytes_per_token(10, 2, 256) / 1024 == gold["kib_per_token_10x2_d256"]
    assert round(100 * oracle.window_fraction(131072), 2) == gold["window_percent_128k"]
    # a request no longer than the two windows is held in BF16 entirely
    assert oracle.window_fraction(100) == 1.0 and oracle.window_fraction(320) == 1.0
    assert oracle.window_fraction(640) == 0.5
    assert oracle.bits_per_element(320, 64) == 16.0
    assert round(oracle.bits_per_element(131072, 128), 2) == gold["bits_per_element"]
    assert round(oracle.bits_per_element(131072, 64, scale_bits=8), 2) == gold["bits_per_element_g64_e4m3"]
    assert oracle.code_bytes_per_token(1, 1, 1) / 2 == gold["bytes_per_code"]
    # per-token record of an 8-KV-head, d=128, G=64 layer: 640 bytes
    assert 8 * oracle.record_bytes(128, 64) == 640
    assert 4 * oracle.record_bytes(256, 128) == 576
    # E4M3 (s, z): 72-byte records, 576 bytes per token of 8 KV heads; the INT2
    # region costs 2 + 16/64 = 2.25 bits per element
    assert 8 * oracle.record_bytes(128, 64, scale_bits=8) == 576
    assert 8 * oracle.record_bytes(128, 64, scale_bits=8) * 8 / (8 * 2 * 128) == 2.25


# --------------------------------------------------------------------------
# cache semantics and attention
# --------------------------------------------------------------------------

def _small_setup(d=64, Hq=4, Hkv=2, G=32, S=4, W=8, clip=0.9, seed=12, R=None):
    cfg = oracle.OracleConfig(d, Hq, Hkv, G, S, W, clip)
    rng = np.random.default_rng(seed)
    if R is None:
        Rk, _ = oracle.build_rotation(oracle.covariance(rng.standard_normal((256, d))), d)
        Rv, _ = oracle.build_rotation(oracle.covariance(rng.standard_normal((256, d))), d)
        Rk = Rk.astype(np.float32)
        Rv = Rv.astype(np.float32)
    else:
        Rk = Rv = R
    return cfg, rng, Rk, Rv


def test_regions():
    S, W = 64, 256
    assert oracle.regions(1024, S, W) == (64, 64, 768, 768, 1024)   # 64 + 704 + 256
    assert oracle.regions(100, S, W) == (64, 64, 64, 64, 100)        # no history
    assert oracle.regions(10, S, W) == (10, 64, 64, 64, 10)          # sink only
    assert oracle.regions(32768, S, W)[2] - 64 == 32448


def test_chunked_append_equals_token_by_token():
    cfg, rng, Rk, Rv = _small_setup()
    L = 40
    k = rng.standard_normal((L, 2, 64)).astype(np.float32) * 3
    v = rng.standard_normal((L, 2, 64)).astype(np.float32)
    pt = rng.permutation(64)[None, :L]
    a = oracle.OracleCache(cfg, 64, 1, Rk, Rv)
    a.append(k, v, [0, L], [0], [0], pt)
    b = oracle.OracleCache(cfg, 64, 1, Rk, Rv)
    pos = 0
    for n in (1, 3, 7, 1, 12, 16):
        b.append(k[pos:pos + n], v[pos:pos + n], [0, n], [pos], [0], pt)
        pos += n
    assert pos == L
    for name in ("kc", "vc", "ks", "kz", "vs", "vz"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name
    assert np.array_equal(a.sink, b.sink)
    hist_hi = oracle.regions(L, cfg.sink, cfg.recent)[2]
    for p in range(hist_hi, L):
        assert np.array_equal(a.ring[0, p % cfg.recent], b.ring[0, p % cfg.recent])


def _textbook_attention(q, K, V):
    d = len(q)
    logits = [sum(q[i] * K[t][i] for i in range(d)) / math.sqrt(d) for t in range(len(K))]
    m = max(logits)
    e = [math.exp(l - m) for l in logits]
    den = sum(e)
    return np.array([sum(e[t] * V[t][i] for t in range(len(K))) / den for i in range(d)])


def test_decode_all_bf16_equals_textbook_attention():
    # L <= S + W: every token is BF16; also checks the GQA-6 head mapping
    d, Hq, Hkv = 16, 12, 2
    cfg = oracle.OracleConfig(d, Hq, Hkv, 16, 4, 8, 0.9)
    rng = np.random.default_rng(13)
    L = 11
    k = rng.standard_normal((L, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((L, Hkv, d)).astype(np.float32) + np.arange(Hkv)[None, :, None] * 10
    cache = oracle.OracleCache(cfg, 16, 1, np.eye(d), np.eye(d))
    cache.append(k, v, [0, L], [0], [0], np.arange(16)[None])
    q = rng.standard_normal((1, Hq, d))
    out = oracle.decode_attention(cache, q, np.arange(16)[None], [L], [0])
    kb = oracle.bf16_round(k).astype(np.float64)
    vb = oracle.bf16_round(v).astype(np.float64)
    for h in range(Hq):
        ref = _textbook_attention(q[0, h], kb[:, h // 6], vb[:, h // 6])
        assert np.abs(out[0, h] - ref).max() <= 1e-12


def test_decode_history_on_grid_equals_textbook_attention():
    # R_K and R_V two different permutations (orthogonal, exact in fp32); history
    # keys and values chosen so that their images under their own rotation lie
    # exactly on the INT2 grid at clip 1.0: then the mixed cache reproduces
    # textbook attention on the original vectors (and a cache that rotated keys
    # by R_V, or values by R_K, would not).
    d, G, S, W = 32, 16, 2, 3
    cfg = oracle.OracleConfig(d, 4, 1, G, S, W, 1.0)
    rng = np.random.default_rng(14)
    Rk = np.eye(d)[:, rng.permutation(d)]      # (x R)[j] = x[perm[j]]
    Rv = np.eye(d)[:, rng.permutation(d)]
    L = 20

    def on_grid(n, R):
        c = rng.integers(0, 4, (n, d))
        c[:, 0::G] = 0
        c[:, 1::G] = 3
        s = 2.0 ** rng.integers(-3, 2, (n, d // G))
        z = rng.integers(-8, 8, (n, d // G)) * 0.25
        y = (z[:, :, None] + c.reshape(n, d // G, G) * s[:, :, None]).reshape(n, d)
        return y @ R.T                          # x with x R = y

    k = on_grid(L, Rk)[:, None, :].astype(np.float32)
    v = on_grid(L, Rv)[:, None, :].astype(np.float32)
    assert np.array_equal(oracle.bf16_round(k), k)
    cache = oracle.OracleCache(cfg, 32, 1, Rk, Rv)
    pt = rng.permutation(32)[None, :L]
    cache.append(k, v, [0, L], [0], [0], pt)
    q = rng.standard_normal((1, 4, d))
    out = oracle.decode_attention(cache, q, pt, [L], [0])
    for h in range(4):
        ref = _textbook_attention(q[0, h], k[:, 0].astype(np.float64), v[:, 0].astype(np.float64))
        assert np.abs(out[0, h] - ref).max() <= 1e-12


def test_split_merge_equals_single_pass():
    cfg, rng, Rk, Rv = _small_setup(d=64, Hq=6, Hkv=2, G=32, S=4, W=8)
    B = 3
    lens = [50, 9, 33]
    cache = oracle.OracleCache(cfg, 200, B, Rk, Rv)
    pt = rng.permutation(200)[:150].reshape(3, 50)
    k = rng.standard_normal((sum(lens), 2, 64)).astype(np.float32) * 2
    v = rng.standard_normal((sum(lens), 2, 64)).astype(np.float32)
    cache.append(k, v, np.cumsum([0] + lens), [0, 0, 0], [0, 1, 2], pt)
    q = rng.standard_normal((B, 6, 64))
    a = oracle.decode_attention(cache, q, pt, lens, [0, 1, 2])
    for chunk in (1, 5, 16, 64):
        b = oracle.decode_attention_split(cache, q, pt, lens, [0, 1, 2], chunk)
        assert np.abs(a - b).max() <= 1e-13


def test_prefill_without_history_equals_textbook_causal_attention():
    # prefix of 5 BF16 tokens (sink 4 + recent 8: no history), chunk of 6
    # queries; GQA 6 mapping; every query sees the prefix and the chunk causally
    d, Hq, Hkv = 16, 12, 2
    cfg = oracle.OracleConfig(d, Hq, Hkv, 16, 4, 8, 0.9)
    rng = np.random.default_rng(21)
    L0, C = 5, 6
    k = rng.standard_normal((L0 + C, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((L0 + C, Hkv, d)).astype(np.float32) + np.arange(Hkv)[None, :, None] * 10
    cache = oracle.OracleCache(cfg, 16, 1, np.eye(d), np.eye(d))
    cache.append(k[:L0], v[:L0], [0, L0], [0], [0], np.arange(16)[None])
    q = rng.standard_normal((C, Hq, d))
    out = oracle.prefill_attention(cache, q, k[L0:], v[L0:], np.arange(16)[None], L0, 0)
    kb = oracle.bf16_round(k).astype(np.float64)
    vb = oracle.bf16_round(v).astype(np.float64)
    for i in range(C):
        for h in range(Hq):
            ref = _textbook_attention(q[i, h], kb[:L0 + i + 1, h // 6], vb[:L0 + i + 1, h // 6])
            assert np.abs(out[i, h] - ref).max() <= 1e-12


def test_prefill_of_one_token_equals_decode_with_a_wider_window():
    # The cache before the append with recent window W, plus the new token at
    # bf16, is the cache after the append with window W + 1: same sink, same
    # history records [S, L0 - W), recent [L0 - W, L0 + 1).
    d, Hq, Hkv, G, S, W = 32, 4, 2, 16, 4, 8
    rng = np.random.default_rng(22)
    Rk, _ = oracle.build_rotation(oracle.covariance(rng.standard_normal((256, d))), d)
    Rv, _ = oracle.build_rotation(oracle.covariance(rng.standard_normal((256, d))), d)
    L0 = 40
    k = (rng.standard_normal((L0 + 1, Hkv, d)) * 3).astype(np.float32)
    v = rng.standard_normal((L0 + 1, Hkv, d)).astype(np.float32)
    pt = rng.permutation(64)[None, :L0 + 1]
    a = oracle.OracleCache(oracle.OracleConfig(d, Hq, Hkv, G, S, W), 64, 1, Rk, Rv)
    a.append(k[:L0], v[:L0], [0, L0], [0], [0], pt)
    wide = oracle.OracleCache(oracle.OracleConfig(d, Hq, Hkv, G, S, W + 1), 64, 1, Rk, Rv)
    wide.append(k, v, [0, L0 + 1], [0], [0], pt)
    q = rng.standard_normal((1, Hq, d))
    got = oracle.prefill_attention(a, q, k[L0:], v[L0:], pt, L0, 0)
    want = oracle.decode_attention(wide, q, pt, [L0 + 1], [0])
    assert np.abs(got - want).max() <= 1e-12

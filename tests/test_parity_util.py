"""Host checks of the parity helpers' rounding-tie bands (no GPU)."""

import numpy as np

from parity_util import ATOL, REL_TIE, RTOL_L2, attn_errors, classify_records, e4m3_near_tie, fp16_near_tie


def test_fp16_near_tie_bands():
    # 1 + 2^-11 is the midpoint between fp16 1.0 and its successor
    mid = np.float32(1.0 + 2.0 ** -11)
    assert fp16_near_tie(mid)
    off = np.float32(mid + 4 * REL_TIE)            # outside the relative band
    assert not fp16_near_tie(off)
    assert fp16_near_tie(off, band=5 * REL_TIE)     # inside an absolute band that covers it
    far = np.float32(1.0 + 2.0 ** -12)              # a quarter step from either neighbour
    assert not fp16_near_tie(far, band=1e-5)


def test_e4m3_near_tie_bands():
    # 1.0625 is the midpoint between E4M3 1.0 and 1.125; 2^-10 between 0 and 2^-9
    for mid in (1.0625, -1.0625, 2.0 ** -10, 432.0):
        assert e4m3_near_tie(np.float32(mid))
        assert not e4m3_near_tie(np.float32(mid * (1 + 4 * REL_TIE)))
    assert not e4m3_near_tie(np.float32(1.03125))        # a quarter step
    assert not e4m3_near_tie(np.float32(464.0))          # saturated range: no tie
    assert e4m3_near_tie(np.float32(1.0625 + 1e-4), band=2e-4)


def _tie_cache(scale_fmt="f16"):
    """An oracle cache with one history token whose K group 0 holds a value at a
    rounding boundary: R = I, clip 1, group min 0 and max 3 give s = 1 and
    z = 0, so channel 1 (y = 0.5) sits exactly on the boundary between codes 0
    and 1 and channel 2 (y = 1.203125) is far from any boundary."""
    import oracle
    d, G = 64, 64
    cfg = oracle.OracleConfig(d, 1, 1, G, sink=0, recent=1, clip_ratio=1.0, scale_fmt=scale_fmt)
    eye = np.eye(d)
    oc = oracle.OracleCache(cfg, 4, 1, eye, eye)
    rng = np.random.default_rng(3)
    x = oracle.bf16_round(rng.uniform(0.25, 2.75, (2, 1, d)).astype(np.float32))
    x[0, 0, 0], x[0, 0, 1], x[0, 0, 2], x[0, 0, 3] = 0.0, 0.5, 1.203125, 3.0
    pt = np.arange(4, dtype=np.int32)[None, :]
    oc.append(x, x, [0, 2], [0], [0], pt, keep_y=True)     # token 0 enters the history
    return oc, d, G


def test_classify_records_excuses_only_boundary_cases():
    # planted on the host, in a copy of the oracle's own records
    from oracle import quant as oq
    oc, d, G = _tie_cache()
    want = oc.records()
    kc, ks, kz, vc, vs, vz = oq.unpack_record(want[0, 0], d, G)
    assert float(ks[0]) == 1.0 and float(kz[0]) == 0.0 and kc[1] == 0 and kc[2] == 1
    assert classify_records(want, oc, [0])["bad"] == 0
    # the code of the tied channel flipped to the other side: a counted tie
    tied = want.copy()
    kc2 = kc.copy()
    kc2[1] = 1
    tied[0, 0] = oq.pack_record(kc2, ks, kz, vc, vs, vz, d, G)
    st = classify_records(tied, oc, [0])
    assert st["bad"] == 0 and st["code_ties"] == 1
    # a code 0.2 away from a boundary flipped: not excused
    wrong = want.copy()
    kc3 = kc.copy()
    kc3[2] = 2
    wrong[0, 0] = oq.pack_record(kc3, ks, kz, vc, vs, vz, d, G)
    st = classify_records(wrong, oc, [0])
    assert st["bad"] == 1 and st["code_ties"] == 0
    # a scale one fp16 step off, with no tie behind it: not excused
    off = want.copy()
    ks4 = ks.copy()
    ks4[0] = np.nextafter(ks4[0], np.float16(2))
    off[0, 0] = oq.pack_record(kc, ks4, kz, vc, vs, vz, d, G)
    st = classify_records(off, oc, [0])
    assert st["bad"] == 1 and st["sz_ties"] == 0


def test_classify_e4m3_slot_records():
    # the same planted cases on E4M3 records held in the slot layout
    from oracle import quant as oq
    oc, d, G = _tie_cache("e4m3")
    want = oc.records()
    kc, ks, kz, vc, vs, vz = oq.unpack_record(want[0, 0], d, G, "e4m3")
    assert float(ks[0]) == 1.0 and float(kz[0]) == 0.0 and kc[1] == 0 and kc[2] == 1
    slots = oc.slot_records()
    assert slots.shape == (4, oc.slot_bytes()) and classify_records(slots, oc, [0])["bad"] == 0
    rb = oc.record_bytes()
    tied = slots.copy()
    kc2 = kc.copy()
    kc2[1] = 1
    tied[0, :rb] = oq.pack_record(kc2, ks, kz, vc, vs, vz, d, G, "e4m3")
    st = classify_records(tied, oc, [0])
    assert st["bad"] == 0 and st["code_ties"] == 1
    off = slots.copy()
    ks4 = ks.copy()
    ks4[0] = np.float16(1.125)                          # one E4M3 step up
    off[0, :rb] = oq.pack_record(kc, ks4, kz, vc, vs, vz, d, G, "e4m3")
    st = classify_records(off, oc, [0])
    assert st["bad"] == 1 and st["sz_ties"] == 0


def test_classify_records_band_is_the_stated_rule():
    # a flipped code is excused only when its quotient lies within 1e-6 of the
    # boundary: the oracle's y of the tied channel is moved 2^-21 (4.8e-7) and
    # 2^-18 (3.8e-6) past u = 0.5, with s = 1 and z = 0 unchanged
    from oracle import quant as oq
    oc, d, G = _tie_cache()
    want = oc.records()
    kc, ks, kz, vc, vs, vz = oq.unpack_record(want[0, 0], d, G)
    kc2 = kc.copy()
    kc2[1] = 1
    flipped = want.copy()
    flipped[0, 0] = oq.pack_record(kc2, ks, kz, vc, vs, vz, d, G)
    ky, vy = oc.ky[0], oc.vy[0]
    for dy, bad in ((2.0 ** -21, 0), (2.0 ** -18, 1)):
        ky2 = ky.copy()
        ky2[0, 1] = np.float32(0.5 + dy)
        st = classify_records(flipped, oc, [0], ora_y={0: (ky2, vy)})
        assert st["bad"] == bad and st["code_ties"] == 1 - bad


def test_attention_error_measures():
    # max-abs over every element and relative L2 over the whole output, against
    # values worked by hand; the bounds are the stated 2e-3 and 1e-3
    want = np.zeros((2, 3, 4))
    want[0, 0, :] = [3.0, 4.0, 0.0, 0.0]                 # |want| = 5
    got = want.copy()
    got[1, 2, 3] = 0.004                                  # one element off by 4e-3
    err, rel = attn_errors(got, want)
    assert err == 0.004 and abs(rel - 0.004 / 5.0) < 1e-15
    got[0, 1, 0] = -0.003
    err, rel = attn_errors(got, want)
    assert err == 0.004 and abs(rel - 0.005 / 5.0) < 1e-15   # sqrt(0.004^2 + 0.003^2) = 0.005
    assert (ATOL, RTOL_L2) == (2e-3, 1e-3)

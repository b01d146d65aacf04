"""Planted mistakes in the oracle must make its pins fail (CPU only).

Each case plants one plausible mistake in the oracle: a dropped term, a wrong
sign, bound or normalisation, a transposed operand, an off-by-one, a wrong
rounding.  It either replaces one oracle function, in every oracle module
that holds it, by a version with the mistake, or hands one oracle module a
numpy whose routine is swapped for the wrong one, so that the oracle's own
code runs with the mistake inside.  The pins that cover the function
(tests/test_oracle_pins.py) then run, and at least one of them must fail.
The oracle's sources are never edited; monkeypatch restores every name after
each case.
"""

import inspect
import sys
import types

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins


def _oracle_modules():
    return [m for k, m in list(sys.modules.items())
            if m is not None and (k == "oracle" or k.startswith("oracle."))]


def _plant(mp, module, name, make):
    """Replace oracle function `name` (defined in `module`) everywhere the
    oracle's modules hold it by make(original)."""
    orig = getattr(module, name)
    mutant = make(orig)
    n = 0
    for mod in _oracle_modules():
        for attr, val in list(vars(mod).items()):
            if val is orig:
                mp.setattr(mod, attr, mutant)
                n += 1
    assert n > 0


class _NumpyWith:
    """numpy with some routines replaced (planted into one oracle module)."""

    def __init__(self, **over):
        self._over = over

    def __getattr__(self, k):
        return self._over[k] if k in self._over else getattr(np, k)


def _plant_np(mp, module, **over):
    mp.setattr(module, "np", _NumpyWith(**over))


def _plant_src(mp, module, old, new):
    """Run `module`'s source with `old` replaced by `new` (in memory: the file is
    only read) and put the mutated module's functions and classes wherever the
    oracle's modules hold the originals."""
    src = inspect.getsource(module)
    assert src.count(old) == 1, old
    mut = types.ModuleType(module.__name__)
    mut.__dict__.update(__name__=module.__name__, __package__="oracle", __file__=module.__file__)
    exec(compile(src.replace(old, new), module.__file__, "exec"), mut.__dict__)
    swaps = {}
    for attr, val in vars(module).items():
        if (inspect.isfunction(val) or inspect.isclass(val)) and val.__module__ == module.__name__:
            swaps[id(val)] = mut.__dict__[attr]
    n = 0
    for mod in _oracle_modules():
        for attr, val in list(vars(mod).items()):
            if id(val) in swaps:
                mp.setattr(mod, attr, swaps[id(val)])
                n += 1
    assert n > 0


def _fails(test_fn):
    try:
        test_fn()
    except Exception:          # an assertion, or an error the mistake causes
        return True
    return False


# --------------------------------------------------------------------------
# mutants
# --------------------------------------------------------------------------

def _hadamard_sign_flip(orig):
    def f(n):
        H = np.array(orig(n), copy=True)
        if n >= 2:
            H[n - 1, n - 1] = -H[n - 1, n - 1]
        return H
    return f


def _eig_ascending(orig):
    def f(C):
        w, U = orig(C)
        return w[::-1].copy(), U[:, ::-1].copy()
    return f


def _eig_sign_flipped(orig):
    def f(C):
        w, U = orig(C)
        U = U.copy()
        U[:, 0] = -U[:, 0]
        return w, U
    return f


def _rotation_transposed(orig):
    def f(*a, **k):
        out = orig(*a, **k)
        if isinstance(out, tuple):
            return (np.ascontiguousarray(out[0].T),) + tuple(out[1:])
        return np.ascontiguousarray(out.T)
    return f


def _rotation_without_bitrev(orig):
    def f(C, d, use_bitrev=True, hadamard_block=None):
        return orig(C, d, use_bitrev=False, hadamard_block=hadamard_block)
    return f


def _block_hadamard_full(orig):
    def f(d, block):
        return orig(d, d)
    return f


def _covariance_n_minus_1(orig):
    def f(X):
        n = np.asarray(X).shape[0]
        return orig(X) * n / max(n - 1, 1)
    return f


def _value_covariance_by_keys(orig):
    def f(S, V):
        S = np.asarray(S)
        return orig(S, V) * S.shape[0] / S.shape[1]
    return f


def _bf16_truncating(orig):
    def f(x):
        x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
        return (x32.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).reshape(x32.shape)
    return f


def _e4m3_saturating_at_240(orig):
    def f(x):
        return orig(np.clip(np.asarray(x, dtype=np.float64), -240.0, 240.0))
    return f


def _ties_away(orig, dtype):
    # round to nearest with ties away from zero: at a tie the two neighbours of
    # x round differently; take the one of larger magnitude
    def f(x):
        xa = np.asarray(x, dtype=dtype)
        up = np.asarray(orig(np.nextafter(xa, np.asarray(np.inf, dtype))), np.float64)
        dn = np.asarray(orig(np.nextafter(xa, np.asarray(-np.inf, dtype))), np.float64)
        r = np.asarray(orig(xa), np.float64)
        tie = (up != dn) & (r != xa.astype(np.float64))
        away = np.where(np.abs(up) >= np.abs(dn), up, dn)
        return np.where(tie, away, r).astype(np.asarray(orig(xa)).dtype)
    return f


def _pack_high_bits_first(orig):
    def f(codes):
        codes = np.asarray(codes, dtype=np.uint8)
        d = codes.shape[-1]
        c = codes.reshape(codes.shape[:-1] + (d // 4, 4)).astype(np.uint16)
        b = (c[..., 0] << 6) | (c[..., 1] << 4) | (c[..., 2] << 2) | c[..., 3]
        return b.astype(np.uint8)
    return f


def _regions_wider_recent(orig):
    def f(L, S, W):
        return orig(L, S, W + 1)
    return f


def _bits_without_windows(orig):
    def f(L, group_size, sink=64, recent=256, scale_bits=16):
        return orig(L, group_size, sink=0, recent=0, scale_bits=scale_bits)
    return f


def _gqa_perm(Hq, g):
    """h2[h]: a head index that the oracle maps to KV head h % Hkv (h2 // g)."""
    Hkv = Hq // g
    return [(h % Hkv) * g + h // Hkv for h in range(Hq)]


def _decode_gqa_interleaved(orig):
    # query head h reads KV head h % Hkv instead of h // g
    def f(cache, q, page_table, seq_lens, req_idx, pairs=None):
        q = np.asarray(q, dtype=np.float64)
        Hq = q.shape[1]
        h2 = _gqa_perm(Hq, cache.cfg.gqa)
        q2 = np.empty_like(q)
        for h in range(Hq):
            q2[:, h2[h]] = q[:, h]
        r = orig(cache, q2, page_table, seq_lens, req_idx,
                 None if pairs is None else [(b, h2[h]) for b, h in pairs])
        out = np.empty_like(r)
        for h in range(Hq):
            out[:, h] = r[:, h2[h]]
        return out
    return f


def _prefill_gqa_interleaved(orig):
    def f(cache, q, k, v, page_table, L0, rq, b=0, heads=None):
        q = np.asarray(q, dtype=np.float64)
        Hq = q.shape[1]
        h2 = _gqa_perm(Hq, cache.cfg.gqa)
        q2 = np.empty_like(q)
        for h in range(Hq):
            q2[:, h2[h]] = q[:, h]
        r = orig(cache, q2, k, v, page_table, L0, rq, b=b,
                 heads=None if heads is None else [h2[h] for h in heads])
        out = np.empty_like(r)
        for h in range(Hq):
            out[:, h] = r[:, h2[h]]
        return out
    return f


def _unpack_reversed(orig):
    def f(packed):
        packed = np.asarray(packed, dtype=np.uint8)
        parts = [(packed >> (2 * (3 - k))) & 3 for k in range(4)]
        out = np.stack(parts, axis=-1)
        return out.reshape(packed.shape[:-1] + (packed.shape[-1] * 4,)).astype(np.uint8)
    return f


def _record_bytes_unpadded(orig):
    def f(head_dim, group_size, scale_bits=16):
        return head_dim // 2 + 2 * 2 * (scale_bits // 8) * (head_dim // group_size)
    return f


def _quantize_into_rotations_swapped(orig):
    # the cache rotates history keys by R_V and values by R_K
    def f(self, slots, Xk, Xv, keep_y=False):
        rk, rv = self.rot_k, self.rot_v
        self.rot_k, self.rot_v = rv, rk
        try:
            return orig(self, slots, Xk, Xv, keep_y)
        finally:
            self.rot_k, self.rot_v = rk, rv
    return f


class _CacheView:
    """A cache whose rotation attribute is seen transposed by the oracle."""

    def __init__(self, cache, which):
        self._c = cache
        self._which = which

    def __getattr__(self, k):
        v = getattr(self._c, k)
        return np.ascontiguousarray(v.T) if k == self._which else v


class _CacheIdentity:
    """A cache whose rotation attribute is seen as the identity by the oracle."""

    def __init__(self, cache, which):
        self._c = cache
        self._which = which

    def __getattr__(self, k):
        v = getattr(self._c, k)
        return np.eye(v.shape[0]) if k == self._which else v


def _attention_without(which):
    def make(orig):
        def f(cache, *a, **k):
            return orig(_CacheIdentity(cache, which), *a, **k)
        return f
    return make


def _attention_with_transposed(which):
    def make(orig):
        def f(cache, *a, **k):
            return orig(_CacheView(cache, which), *a, **k)
        return f
    return make


# --------------------------------------------------------------------------
# cases: (id, planting function, pins that must not all pass)
# --------------------------------------------------------------------------

R = oracle.rotation
Q = oracle.quant
A = oracle.attention
P = oracle.prefill
C = oracle.cache
ACC = oracle.accounting

CASES = [
    ("hadamard: one entry of the wrong sign",
     lambda mp: _plant(mp, R, "hadamard", _hadamard_sign_flip),
     [pins.test_hadamard_matches_golden_and_closed_form, pins.test_hadamard_256_exactly_orthogonal_in_fp32]),
    ("bit reversal left out (identity permutation)",
     lambda mp: _plant(mp, R, "bitrev_indices", lambda o: (lambda d: np.arange(d))),
     [pins.test_bitrev_golden_and_involution]),
    ("eigenvectors in ascending order",
     lambda mp: _plant(mp, R, "eig_desc", _eig_ascending),
     [pins.test_eig_desc_diagonal_is_sorting_permutation_and_signs, pins.test_eig_desc_two_by_two_closed_form]),
    ("eigenvector sign rule broken",
     lambda mp: _plant(mp, R, "eig_desc", _eig_sign_flipped),
     [pins.test_eig_desc_diagonal_is_sorting_permutation_and_signs, pins.test_eig_desc_two_by_two_closed_form]),
    ("rotation returned transposed",
     lambda mp: _plant(mp, R, "build_rotation", _rotation_transposed),
     [pins.test_rotation_is_orthogonal_and_factorises, pins.test_rotation_without_covariance_is_the_pages_hadamard]),
    ("P_br dropped from the rotation",
     lambda mp: _plant(mp, R, "build_rotation", _rotation_without_bitrev),
     [pins.test_rotation_without_covariance_is_the_pages_hadamard,
      pins.test_bitrev_spreads_every_importance_block_over_every_group]),
    ("block Hadamard built at full size",
     lambda mp: _plant(mp, R, "block_hadamard", _block_hadamard_full),
     [pins.test_block_hadamard_closed_form_and_orthogonality,
      pins.test_bitrev_spreads_every_importance_block_over_every_group]),
    ("covariance normalised by N - 1",
     lambda mp: _plant(mp, R, "covariance", _covariance_n_minus_1),
     [pins.test_covariances_against_explicit_sums]),
    ("value covariance normalised by the key count",
     lambda mp: _plant(mp, R, "value_covariance", _value_covariance_by_keys),
     [pins.test_covariances_against_explicit_sums]),
    ("bf16 rounding truncates",
     lambda mp: _plant(mp, Q, "bf16_round", _bf16_truncating),
     [pins.test_bf16_round_matches_torch]),
    ("bf16 rounding with ties away from zero",
     lambda mp: _plant(mp, Q, "bf16_round", lambda o: _ties_away(o, np.float32)),
     [pins.test_bf16_round_matches_torch]),
    ("E4M3 rounding with ties away from zero",
     lambda mp: _plant(mp, Q, "e4m3_round", lambda o: _ties_away(o, np.float32)),
     [pins.test_e4m3_rounding_matches_torch]),
    ("E4M3 saturates at 240",
     lambda mp: _plant(mp, Q, "e4m3_round", _e4m3_saturating_at_240),
     [pins.test_e4m3_rounding_matches_torch]),
    ("codes rounded down instead of to nearest",
     lambda mp: _plant_np(mp, Q, rint=np.floor),
     [pins.test_quantiser_code_is_the_nearest_level_brute_force, pins.test_quantiser_exact_grid_round_trip]),
    ("codes at an exact half rounded away from zero",
     lambda mp: _plant_np(mp, Q, rint=lambda x: np.sign(x) * np.floor(np.abs(x) + 0.5)),
     [pins.test_quantiser_code_is_the_nearest_level_brute_force, pins.test_quantiser_exact_grid_round_trip,
      pins.test_quantiser_ties_round_to_even]),
    ("codes clamped to [0, 2]",
     lambda mp: _plant_np(mp, Q, clip=lambda x, a, b: np.clip(x, a, 2.0)),
     [pins.test_quantiser_code_is_the_nearest_level_brute_force, pins.test_quantiser_exact_grid_round_trip]),
    ("scale and zero stored at bf16 instead of fp16",
     lambda mp: _plant(mp, Q, "_round_scale",
                       lambda o: (lambda x, fmt: Q.bf16_round(np.asarray(x, np.float32)).astype(np.float16)
                                  if fmt == "f16" else o(x, fmt))),
     [pins.test_quantiser_code_is_the_nearest_level_brute_force, pins.test_quantiser_exact_grid_round_trip]),
    ("codes packed high bits first",
     lambda mp: _plant(mp, Q, "pack_codes", _pack_high_bits_first),
     [pins.test_packing_golden_and_round_trip, pins.test_record_round_trip_and_size]),
    ("recent window one token wider",
     lambda mp: _plant(mp, C, "regions", _regions_wider_recent),
     [pins.test_regions]),
    ("softmax scale 1/sqrt(d) dropped",
     lambda mp: _plant_np(mp, A, sqrt=lambda x: 1.0),
     [pins.test_decode_all_bf16_equals_textbook_attention, pins.test_decode_history_on_grid_equals_textbook_attention]),
    ("R_V applied where R_Vᵀ belongs",
     lambda mp: _plant(mp, A, "decode_attention", _attention_with_transposed("rot_v")),
     [pins.test_decode_history_on_grid_equals_textbook_attention, pins.test_rotation_invariance_of_logits_and_attention]),
    ("query rotated by R_Kᵀ instead of R_K",
     lambda mp: _plant(mp, A, "decode_attention", _attention_with_transposed("rot_k")),
     [pins.test_decode_history_on_grid_equals_textbook_attention, pins.test_rotation_invariance_of_logits_and_attention]),
    ("split-K partials merged without R_Vᵀ's transpose",
     lambda mp: _plant(mp, A, "decode_attention_split", _attention_with_transposed("rot_v")),
     [pins.test_split_merge_equals_single_pass]),
    ("prefill's causal mask lets a query see the next token",
     lambda mp: _plant_np(mp, P, tril=lambda x: np.tril(x, 1)),
     [pins.test_prefill_without_history_equals_textbook_causal_attention]),
    ("prefill's softmax scale dropped",
     lambda mp: _plant_np(mp, P, sqrt=lambda x: 1.0),
     [pins.test_prefill_without_history_equals_textbook_causal_attention,
      pins.test_prefill_of_one_token_equals_decode_with_a_wider_window]),
    ("Hadamard factor not normalised",
     lambda mp: _plant(mp, R, "block_hadamard", lambda o: (lambda d, block: o(d, block) * np.sqrt(block))),
     [pins.test_block_hadamard_closed_form_and_orthogonality, pins.test_rotation_is_orthogonal_and_factorises]),
    ("eigenvectors returned as rows",
     lambda mp: _plant(mp, R, "eig_desc", lambda o: (lambda C: (o(C)[0], o(C)[1].T.copy()))),
     [pins.test_eig_desc_reconstructs_random_covariance, pins.test_eig_desc_two_by_two_closed_form]),
    ("covariance of centred rows",
     lambda mp: _plant(mp, R, "covariance",
                       lambda o: (lambda X: o(np.asarray(X, np.float64) - np.asarray(X, np.float64).mean(axis=0)))),
     [pins.test_covariances_against_explicit_sums]),
    ("dequantisation with scale and zero swapped",
     lambda mp: _plant(mp, Q, "dequantize_rows", lambda o: (lambda c, s, z: o(c, z, s))),
     [pins.test_quantiser_exact_grid_round_trip, pins.test_quantiser_flat_group]),
    ("codes unpacked high bits first",
     lambda mp: _plant(mp, Q, "unpack_codes", _unpack_reversed),
     [pins.test_packing_golden_and_round_trip, pins.test_record_round_trip_and_size]),
    ("records not padded",
     lambda mp: _plant(mp, ACC, "record_bytes", _record_bytes_unpadded),
     [pins.test_accounting_matches_pages, pins.test_record_round_trip_and_size]),
    ("sink one token short",
     lambda mp: _plant(mp, C, "regions", lambda o: (lambda L, S, W: o(L, max(S - 1, 0), W))),
     [pins.test_regions]),
    ("query head h reads KV head h mod Hkv (decode)",
     lambda mp: _plant(mp, A, "decode_attention", _decode_gqa_interleaved),
     [pins.test_decode_all_bf16_equals_textbook_attention, pins.test_decode_history_on_grid_equals_textbook_attention]),
    ("query head h reads KV head h mod Hkv (prefill)",
     lambda mp: _plant(mp, P, "prefill_attention", _prefill_gqa_interleaved),
     [pins.test_prefill_without_history_equals_textbook_causal_attention,
      pins.test_prefill_of_one_token_equals_decode_with_a_wider_window]),
    ("prefill's chunk keys and values not rounded to bf16",
     lambda mp: mp.setattr(P, "bf16_round", lambda x: np.asarray(x, np.float32)),
     [pins.test_prefill_without_history_equals_textbook_causal_attention,
      pins.test_prefill_of_one_token_equals_decode_with_a_wider_window]),
    ("history keys rotated by R_V and values by R_K",
     lambda mp: mp.setattr(C.OracleCache, "_quantize_into",
                           _quantize_into_rotations_swapped(C.OracleCache._quantize_into)),
     [pins.test_decode_history_on_grid_equals_textbook_attention, pins.test_chunked_append_equals_token_by_token,
      pins.test_prefill_of_one_token_equals_decode_with_a_wider_window]),
    ("positions entering the history shifted by one",
     lambda mp: _plant_np(mp, C, arange=lambda a, b: np.arange(a + 1, b + 1)),
     [pins.test_decode_history_on_grid_equals_textbook_attention, pins.test_chunked_append_equals_token_by_token,
      pins.test_prefill_of_one_token_equals_decode_with_a_wider_window]),
    ("clip ratio ignored",
     lambda mp: _plant(mp, Q, "quantize_rows",
                       lambda o: (lambda Y, G, r, scale_fmt="f16": o(Y, G, 1.0, scale_fmt))),
     [pins.test_quantiser_code_is_the_nearest_level_brute_force]),
    ("rows rotated by Rᵀ",
     lambda mp: _plant(mp, Q, "rotate_rows", lambda o: (lambda X, Rm: o(X, np.asarray(Rm).T))),
     [pins.test_decode_history_on_grid_equals_textbook_attention, pins.test_chunked_append_equals_token_by_token,
      pins.test_rotation_invariance_of_logits_and_attention]),
    ("history output not rotated back by R_Vᵀ (decode)",
     lambda mp: _plant(mp, A, "decode_attention", _attention_without("rot_v")),
     [pins.test_decode_history_on_grid_equals_textbook_attention]),
    ("history logits against the unrotated query (decode)",
     lambda mp: _plant(mp, A, "decode_attention", _attention_without("rot_k")),
     [pins.test_decode_history_on_grid_equals_textbook_attention]),
    ("history output not rotated back by R_Vᵀ (prefill)",
     lambda mp: _plant(mp, P, "prefill_attention", _attention_without("rot_v")),
     [pins.test_prefill_of_one_token_equals_decode_with_a_wider_window]),
    ("history logits against the unrotated query (prefill)",
     lambda mp: _plant(mp, P, "prefill_attention", _attention_without("rot_k")),
     [pins.test_prefill_of_one_token_equals_decode_with_a_wider_window]),
    ("bits per element without the BF16 windows",
     lambda mp: _plant(mp, ACC, "bits_per_element", _bits_without_windows),
     [pins.test_accounting_matches_pages]),
]


# Source-level mistakes: (module, expression as written, expression with the
# mistake, pins).  Pins of each module:
ROT_PINS = [pins.test_hadamard_matches_golden_and_closed_form, pins.test_bitrev_golden_and_involution,
            pins.test_eig_desc_two_by_two_closed_form, pins.test_eig_desc_diagonal_is_sorting_permutation_and_signs,
            pins.test_eig_desc_reconstructs_random_covariance, pins.test_rotation_without_covariance_is_the_pages_hadamard,
            pins.test_rotation_is_orthogonal_and_factorises, pins.test_block_hadamard_closed_form_and_orthogonality,
            pins.test_bitrev_spreads_every_importance_block_over_every_group, pins.test_covariances_against_explicit_sums]
QUANT_PINS = [pins.test_bf16_round_matches_torch, pins.test_e4m3_rounding_matches_torch,
              pins.test_quantiser_exact_grid_round_trip, pins.test_quantiser_e4m3_exact_grid_round_trip,
              pins.test_quantiser_e4m3_code_is_the_nearest_level_brute_force,
              pins.test_quantiser_code_is_the_nearest_level_brute_force, pins.test_quantiser_ties_round_to_even,
              pins.test_quantiser_flat_group, pins.test_packing_golden_and_round_trip,
              pins.test_record_round_trip_and_size, pins.test_e4m3_record_and_slot_layout]
CACHE_PINS = [pins.test_regions, pins.test_chunked_append_equals_token_by_token,
              pins.test_decode_all_bf16_equals_textbook_attention,
              pins.test_decode_history_on_grid_equals_textbook_attention,
              pins.test_prefill_of_one_token_equals_decode_with_a_wider_window]
ATT_PINS = [pins.test_decode_all_bf16_equals_textbook_attention,
            pins.test_decode_history_on_grid_equals_textbook_attention, pins.test_split_merge_equals_single_pass,
            pins.test_rotation_invariance_of_logits_and_attention,
            pins.test_prefill_of_one_token_equals_decode_with_a_wider_window]
PF_PINS = [pins.test_prefill_without_history_equals_textbook_causal_attention,
           pins.test_prefill_of_one_token_equals_decode_with_a_wider_window]
ACC_PINS = [pins.test_accounting_matches_pages, pins.test_record_round_trip_and_size]

SRC_CASES = [
    (R, "h = np.block([[h, h], [h, -h]])", "h = np.block([[h, h], [-h, h]])", ROT_PINS),
    (R, "r |= 1 << (nbits - 1 - b)", "r |= 1 << (nbits - 1 - b) if b else 0", ROT_PINS),
    (R, 'order = np.argsort(-w, kind="stable")', 'order = np.argsort(w, kind="stable")', ROT_PINS),
    (R, "if col[i] < 0:", "if col[i] > 0:", ROT_PINS),
    (R, "M = M[:, bitrev_indices(d)]", "M = M[bitrev_indices(d), :]", ROT_PINS),
    (R, "M = U @ block_hadamard(d, block)", "M = block_hadamard(d, block) @ U", ROT_PINS),
    (R, "Hb = hadamard(block) / np.sqrt(block)", "Hb = hadamard(block) / block", ROT_PINS),
    (R, "return X.T @ X / X.shape[0]", "return X.T @ X / X.shape[1]", ROT_PINS),
    (Q, "lo = (r * mn).astype(np.float32)", "lo = mn.astype(np.float32)", QUANT_PINS),
    (Q, "/ np.float32(3.0)).astype(np.float32)", "/ np.float32(4.0)).astype(np.float32)", QUANT_PINS),
    (Q, "z16 = _round_scale(lo, scale_fmt)", "z16 = _round_scale(hi, scale_fmt)", QUANT_PINS),
    (Q, "c = np.where(s_f == 0.0, 0.0, c)", "c = np.where(s_f == 0.0, 1.0, c)", QUANT_PINS),
    (Q, "return (s * c + z).reshape(n, d)", "return (s * c - z).reshape(n, d)", QUANT_PINS),
    (Q, "(c[..., 1] << 2) | (c[..., 2] << 4)", "(c[..., 2] << 2) | (c[..., 1] << 4)", QUANT_PINS),
    (Q, "raw = d // 2 + 2 * pb * ng", "raw = d // 2 + pb * ng", QUANT_PINS),
    (Q, "e = np.maximum(ex - 1, -6)", "e = np.maximum(ex - 1, -7)", QUANT_PINS),
    (Q, "r = np.minimum(r, 448.0)", "r = np.minimum(r, 480.0)", QUANT_PINS),
    (Q, "exp_field = np.where(normal, e + 7, 0)", "exp_field = np.where(normal, e + 8, 0)", QUANT_PINS),
    (Q, "np.ldexp(1.0 + m / 8.0, ef - 7)", "np.ldexp(1.0 + m / 8.0, ef - 8)", QUANT_PINS),
    (Q, "out[..., :flat.shape[-1]] = flat", "out[..., slot_size - flat.shape[-1]:] = flat", QUANT_PINS),
    (Q, "return (raw + 15) // 16 * 16", "return (raw + 7) // 8 * 8", QUANT_PINS),
    (Q, "return (x32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)",
     "return (x32.view(np.uint32) >> np.uint32(15)).astype(np.uint16)", QUANT_PINS + CACHE_PINS),
    (ACC, "return num_layers * num_kv_heads * head_dim * 2 * 0.25", "return num_layers * num_kv_heads * head_dim * 0.25",
     ACC_PINS),
    (ACC, "return min(L, sink + recent) / L", "return (sink + recent) / L", ACC_PINS),
    (C, "old = pos < L0", "old = pos <= L0", CACHE_PINS),
    (C, "Xk[old] = self.ring[rq, pos[old] % W, :, 0, :]", "Xk[old] = self.ring[rq, (pos[old] + 1) % W, :, 0, :]",
     CACHE_PINS),
    (C, "self.ring[rq, p % W, :, 1, :] = xv[p - L0]", "self.ring[rq, p % W, :, 1, :] = xk[p - L0]", CACHE_PINS),
    (C, "xv = bf16_round(v[c0:c1])", "xv = np.asarray(v[c0:c1], np.float32)", CACHE_PINS),
    (C, "hist_hi = max(S, L - W)", "hist_hi = max(S, L - W + 1)", CACHE_PINS),
    (C, "Yv = rotate_rows(Xv.reshape(n * H, d), self.rot_v)", "Yv = rotate_rows(Xv.reshape(n * H, d), self.rot_k)",
     CACHE_PINS),
    (A, "den = ep.sum() + eh.sum()", "den = ep.sum()", ATT_PINS),
    (A, "lp = (Kp @ qv) * scale\n            lh", "lp = (Kp @ qr) * scale\n            lh", ATT_PINS),
    (A, "den = sum(np.exp(p[0] - M) * p[1] for p in parts)", "den = sum(p[1] for p in parts)", ATT_PINS),
    (A, "o_rot = sum((np.exp(p[0] - M) * p[2] for p in parts if p[3]),", "o_rot = sum((p[2] for p in parts if p[3]),",
     ATT_PINS),
    (A, "Kp.append(cache.ring[rq, pos % W, kvh, 0, :].astype(np.float64))",
     "Kp.append(cache.ring[rq, pos % W, kvh, 1, :].astype(np.float64))", ATT_PINS),
    (P, "causal = np.tril(np.ones((C, C), dtype=bool))", "causal = np.tril(np.ones((C, C), dtype=bool), -1)",
     PF_PINS),
    (P, "den = ep.sum(axis=1) + eh.sum(axis=1) + ec.sum(axis=1)", "den = ep.sum(axis=1) + ec.sum(axis=1)", PF_PINS),
    (P, "num = ep @ Vp + ec @ vc[:, kvh, :]", "num = ep @ Vp + ec @ kc[:, kvh, :]", PF_PINS),
    (ACC, "raw = head_dim // 2 + 2 * 2 * (scale_bits // 8) * ng", "raw = head_dim // 4 + 2 * 2 * (scale_bits // 8) * ng",
     ACC_PINS),
    (ACC, "(2.0 + 2.0 * scale_bits / group_size)", "(2.0 + scale_bits / group_size)", ACC_PINS),
]


@pytest.mark.parametrize("case", SRC_CASES, ids=["%s: %s" % (c[0].__name__.split(".")[-1], c[2]) for c in SRC_CASES])
def test_source_mistake_fails_a_pin(case, monkeypatch):
    module, old, new, covering = case
    _plant_src(monkeypatch, module, old, new)
    assert any(_fails(t) for t in covering), "no pin caught the planted mistake"


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_planted_mistake_fails_a_pin(case, monkeypatch):
    _, plant, covering = case
    plant(monkeypatch)
    assert any(_fails(t) for t in covering), "no pin caught the planted mistake"


def test_pins_pass_without_a_planted_mistake():
    for t in {t for _, _, ts in CASES for t in ts}:
        t()
